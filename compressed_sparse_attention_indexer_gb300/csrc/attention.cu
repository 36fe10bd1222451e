// Steps (c) + (d): gather the rows a query reads and attend over them.
//
// hw-native-sys/pypto-lib:
//  - "Fix: port the DeepSeek-V4 MoE, hc_pre and prefill fixes to DSpark", PR
//    description: a query reads at most WIN + min(max_visible_cmp, IDX_TOPK)
//    sparse rows (window rows + the indexer's selection);
//  - "Perf: skip redundant CSA scoring and fuse gather unpack", PR
//    description: gathered rows are read straight into their consumer (here:
//    shared-memory tiles of the attention kernel; no packed intermediate);
//  - "Perf: fuse HCA merge, inverse RoPE, and packing", PR description: the
//    raw (window) and compressed softmax streams are merged, then inverse RoPE
//    is applied, in one kernel.
//
// Rows are shared by all heads: the score of head h on row u uses all D row
// dims, the value is the first V dims.  Streams, in fixed order: window (raw
// rows pos-nwin+1..pos), compressed (the Top-K rows), heavy compression (all
// vis2 rows, when enabled).  Each stream keeps its own running max / sum /
// output; when a stream ends it is folded into the merged result by a
// log-sum-exp merge.  The merged output's last R dims are rotated back by
// -pos * base^(-2i/R) on interleaved pairs.
//
// Tensor-core path (bf16, H = 64, D = 576, V = 512): one CTA per (query, half
// of the heads).  Rows arrive in 64-row tiles through a two-stage cp.async
// ring (index lookup and bounds checks done once per row), swizzled so that
// ldmatrix reads are conflict free.  S = Q.R^T and O += P.V run on warp MMA
// with fp32 accumulators; P is rounded to bf16 for the second product.
//
// SIMT path: any shape / dtype, one warp per head, fp32 arithmetic.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include "csa_internal.cuh"
#include "ptx.cuh"

namespace csa {

namespace {

constexpr int kAttnThreads = 256;
constexpr int kHPC = 32;                  // heads per CTA
constexpr int kTR = 64;                   // rows per tile
constexpr int kRowBytes = kTcD * 2;       // 1152
constexpr int kRowChunks = kRowBytes / 16;  // 72
constexpr int kQsBytes = kHPC * kRowBytes;  // 36864
constexpr int kTileBytes = kTR * kRowBytes; // 73728
constexpr int kPsBytes = 2 * 16 * kTR * 2;  // 4096
constexpr int kAttnSmem = kQsBytes + 2 * kTileBytes + kPsBytes;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnShared {
  float red_max[2][4][16];
  float red_l[2][4][16];
  const __nv_bfloat16* rowptr[2][kTR];
  float2 rope[32];
};

__device__ __forceinline__ const __nv_bfloat16* row_pointer(const DevBatch& b, const QueryPlan& p,
                                                            int bi, int q, int K,
                                                            const int* __restrict__ topk_idx,
                                                            int sid, int i, int* status) {
  int64_t gr;
  const __nv_bfloat16* base;
  int64_t stride, rows;
  if (sid == 0) {
    gr = raw_row(b, bi, p.pos - p.nwin + 1 + i);
    base = static_cast<const __nv_bfloat16*>(b.raw); stride = b.raw_stride; rows = b.raw_rows;
  } else if (sid == 1) {
    const int j = topk_idx[(int64_t)q * K + i];
    if (j < 0 || j >= p.vis) {
      set_status(status, kStatusBadIndex);
      return nullptr;
    }
    gr = cmp_row(b, bi, j);
    base = static_cast<const __nv_bfloat16*>(b.cmp); stride = b.cmp_stride; rows = b.cmp_rows;
  } else {
    gr = hca_row(b, bi, i);
    base = static_cast<const __nv_bfloat16*>(b.hca); stride = b.hca_stride; rows = b.hca_rows;
  }
  if (gr < 0 || gr >= rows) {
    set_status(status, kStatusBadIndex);
    return nullptr;
  }
  return base + gr * stride;
}

// The query's plan, with its Top-K count taken from topk_cnt (written by the
// Top-K kernel or supplied by the caller).  A count outside [0, min(vis, K)]
// is clamped and reported, as is a bad length.
__device__ __forceinline__ QueryPlan attn_plan(const DevCfg& c, const DevBatch& b, int q,
                                               const int* __restrict__ topk_cnt, int* status,
                                               bool report) {
  const int bi = q / b.S;
  QueryPlan p = query_plan(c, b.S, b.ctx_len[bi], q - bi * b.S, 0);
  if (p.flags & kPlanBad) {
    if (report) set_status(status, kStatusBadIndex);
    return p;
  }
  int ci = topk_cnt[q];
  if (ci < 0 || ci > p.cnt) {
    if (report) set_status(status, kStatusBadIndex);
    ci = ci < 0 ? 0 : p.cnt;
  }
  p.cnt = ci;
  return p;
}

__global__ void __launch_bounds__(kAttnThreads, 1)
    attn_tc_kernel(DevCfg c, DevBatch b, Workspace ws, const int* __restrict__ topk_idx,
                   const int* __restrict__ topk_cnt, __nv_bfloat16* __restrict__ out,
                   float* __restrict__ lse_out) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* Qs = smem;
  uint8_t* Rs = Qs + kQsBytes;
  uint8_t* Ps = Rs + 2 * kTileBytes;
  __shared__ AttnShared sh;

  const int q = blockIdx.x >> 1, hh = blockIdx.x & 1;
  pdl_wait();
  pdl_trigger();
  const QueryPlan p = attn_plan(c, b, q, topk_cnt, ws.status, threadIdx.x == 0 && hh == 0);
  const int bi = q / b.S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t4 = lane & 3;
  const int mt = warp & 1;       // 16-head tile of this warp
  const int rg = warp >> 1;      // QK: 16-row group of the tile; PV: 128-column quarter
  const int head0 = hh * kHPC + mt * 16;

  if (p.flags & kPlanBad) {
    for (int v = tid; v < kHPC * kTcV / 2; v += kAttnThreads)
      reinterpret_cast<uint32_t*>(out + ((int64_t)q * kTcH + hh * kHPC) * kTcV)[v] = 0u;
    if (lse_out && tid < kHPC) lse_out[(int64_t)q * kTcH + hh * kHPC + tid] = -INFINITY;
    return;
  }

  const int ns[3] = {p.nwin, p.cnt, p.vis2};
  const int nt0 = (ns[0] + kTR - 1) / kTR, nt1 = (ns[1] + kTR - 1) / kTR,
            nt2 = (ns[2] + kTR - 1) / kTR;
  const int Tt = nt0 + nt1 + nt2;

  if (tid < 32) sh.rope[tid] = rope_cos_sin((double)p.pos, c.rope_theta[tid]);

  auto tile_stream = [&](int t, int& sid, int& lt) {
    if (t < nt0) { sid = 0; lt = t; }
    else if (t < nt0 + nt1) { sid = 1; lt = t - nt0; }
    else { sid = 2; lt = t - nt0 - nt1; }
  };
  auto prep_rows = [&](int t) {
    if (tid < kTR) {
      int sid, lt;
      tile_stream(t, sid, lt);
      const int i = lt * kTR + tid;
      sh.rowptr[t & 1][tid] =
          i < ns[sid] ? row_pointer(b, p, bi, q, c.K, topk_idx, sid, i, ws.status) : nullptr;
    }
  };
  const __nv_bfloat16* any_ptr = static_cast<const __nv_bfloat16*>(b.q);
  auto issue_rows = [&](int t) {
    uint8_t* dst0 = Rs + (t & 1) * kTileBytes;
#pragma unroll 6
    for (int i = 0; i < kTR * kRowChunks / kAttnThreads; ++i) {
      const int id = tid + i * kAttnThreads;
      const int row = id / kRowChunks, ch = id - row * kRowChunks;
      const __nv_bfloat16* rp = sh.rowptr[t & 1][row];
      cp_async16(smem_u32(dst0 + row * kRowBytes + ((ch ^ (row & 7)) << 4)),
                 rp ? (const void*)(rp + ch * 8) : (const void*)any_ptr, rp ? 16 : 0);
    }
  };

  prep_rows(0);
  __syncthreads();
  {
    const __nv_bfloat16* qsrc =
        static_cast<const __nv_bfloat16*>(b.q) + ((int64_t)q * kTcH + hh * kHPC) * kTcD;
    for (int id = tid; id < kHPC * kRowChunks; id += kAttnThreads) {
      const int row = id / kRowChunks, ch = id - row * kRowChunks;
      cp_async16(smem_u32(Qs + row * kRowBytes + ((ch ^ (row & 7)) << 4)),
                 qsrc + row * kTcD + ch * 8, 16);
    }
    issue_rows(0);
    cp_async_commit();
  }

  const float sc2 = c.scale * kLog2e;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.f, 0.f};
  float o[16][4], om[16][4];
  float lse_m[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int j = 0; j < 16; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = om[j][e] = 0.f;

  for (int t = 0; t < Tt; ++t) {
    if (t + 1 < Tt) prep_rows(t + 1);
    __syncthreads();
    if (t + 1 < Tt) issue_rows(t + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    int sid, lt;
    tile_stream(t, sid, lt);
    const uint8_t* Rt = Rs + (t & 1) * kTileBytes;

    // ---- S = Q . R^T for 16 heads x 16 rows over all 576 dims
    float s[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
    {
      const int qrow = mt * 16 + (lane & 15);
      const int rrow = rg * 16 + ((lane >> 4) << 3) + (lane & 7);
      const uint8_t* qb = Qs + qrow * kRowBytes;
      const uint8_t* rb = Rt + rrow * kRowBytes;
#pragma unroll 6
      for (int kk = 0; kk < kTcD / 16; ++kk) {
        uint32_t a[4], r0, r1, r2, r3;
        const int qc = 2 * kk + (lane >> 4);
        ldsm_x4(smem_u32(qb + ((qc ^ (qrow & 7)) << 4)), a[0], a[1], a[2], a[3]);
        const int rc = 2 * kk + ((lane >> 3) & 1);
        ldsm_x4(smem_u32(rb + ((rc ^ (rrow & 7)) << 4)), r0, r1, r2, r3);
        mma_bf16_16816(s[0], a, r0, r1);
        mma_bf16_16816(s[1], a, r2, r3);
      }
    }
    // scale to log2 units, mask rows that do not exist
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = rg * 16 + nt * 8 + 2 * t4 + (e & 1);
        const bool ok = sh.rowptr[t & 1][row] != nullptr;
        s[nt][e] = ok ? s[nt][e] * sc2 : -INFINITY;
      }
      mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    if (t4 == 0) {
      sh.red_max[mt][rg][g] = mx0;
      sh.red_max[mt][rg][g + 8] = mx1;
    }
    __syncthreads();
    float tm0 = sh.red_max[mt][0][g], tm1 = sh.red_max[mt][0][g + 8];
#pragma unroll
    for (int r = 1; r < 4; ++r) {
      tm0 = fmaxf(tm0, sh.red_max[mt][r][g]);
      tm1 = fmaxf(tm1, sh.red_max[mt][r][g + 8]);
    }
    const float mn0 = fmaxf(m_run[0], tm0), mn1 = fmaxf(m_run[1], tm1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2f(m_run[0] - mu0), al1 = exp2f(m_run[1] - mu1);
    m_run[0] = mn0;
    m_run[1] = mn1;
    float ps0 = 0.f, ps1 = 0.f;
    uint8_t* Pm = Ps + mt * (16 * kTR * 2);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const float p0 = exp2f(s[nt][0] - mu0), p1 = exp2f(s[nt][1] - mu0);
      const float p2 = exp2f(s[nt][2] - mu1), p3 = exp2f(s[nt][3] - mu1);
      ps0 += p0 + p1;
      ps1 += p2 + p3;
      const int chunk = rg * 2 + nt;
      *reinterpret_cast<uint32_t*>(Pm + g * 128 + ((chunk ^ (g & 7)) << 4) + 4 * t4) =
          pack_bf16x2(p0, p1);
      *reinterpret_cast<uint32_t*>(Pm + (g + 8) * 128 + ((chunk ^ ((g + 8) & 7)) << 4) + 4 * t4) =
          pack_bf16x2(p2, p3);
    }
    l_run[0] = l_run[0] * al0 + ps0;
    l_run[1] = l_run[1] * al1 + ps1;
    __syncthreads();

    // ---- O[16 heads x 128 cols] = O * alpha + P . V
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      o[j][0] *= al0; o[j][1] *= al0;
      o[j][2] *= al1; o[j][3] *= al1;
    }
#pragma unroll
    for (int kk = 0; kk < kTR / 16; ++kk) {
      uint32_t a[4];
      {
        const int prow = lane & 15;
        const int pc = 2 * kk + (lane >> 4);
        ldsm_x4(smem_u32(Pm + prow * 128 + ((pc ^ (prow & 7)) << 4)), a[0], a[1], a[2], a[3]);
      }
      const int vrow = kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
      const uint8_t* vb = Rt + vrow * kRowBytes;
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        const int vc = rg * 16 + np * 2 + (lane >> 4);
        uint32_t r0, r1, r2, r3;
        ldsm_x4_trans(smem_u32(vb + ((vc ^ (vrow & 7)) << 4)), r0, r1, r2, r3);
        mma_bf16_16816(o[2 * np], a, r0, r1);
        mma_bf16_16816(o[2 * np + 1], a, r2, r3);
      }
    }

    // ---- end of a stream: fold it into the merged result (LSE merge)
    const bool last_of_stream = (t + 1 == Tt) || (t + 1 == nt0) || (t + 1 == nt0 + nt1);
    if (last_of_stream) {
      float l0 = l_run[0], l1 = l_run[1];
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      if (t4 == 0) {
        sh.red_l[mt][rg][g] = l0;
        sh.red_l[mt][rg][g + 8] = l1;
      }
      __syncthreads();
      const float L0 = ((sh.red_l[mt][0][g] + sh.red_l[mt][1][g]) + sh.red_l[mt][2][g]) + sh.red_l[mt][3][g];
      const float L1 = ((sh.red_l[mt][0][g + 8] + sh.red_l[mt][1][g + 8]) + sh.red_l[mt][2][g + 8]) +
                       sh.red_l[mt][3][g + 8];
      const float Ls[2] = {L0, L1};
#pragma unroll
      for (int hi = 0; hi < 2; ++hi) {
        if (Ls[hi] > 0.f) {
          const float lse_s = m_run[hi] + log2f(Ls[hi]);
          const float nl = fmaxf(lse_m[hi], lse_s);
          const float wa = exp2f(lse_m[hi] - nl), wb = exp2f(lse_s - nl);
          const float tot = wa + wb;
          const float fa = wa / tot, fb = wb / (tot * Ls[hi]);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            om[j][2 * hi] = om[j][2 * hi] * fa + o[j][2 * hi] * fb;
            om[j][2 * hi + 1] = om[j][2 * hi + 1] * fa + o[j][2 * hi + 1] * fb;
          }
          lse_m[hi] = nl + log2f(tot);
        }
        m_run[hi] = -INFINITY;
        l_run[hi] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 16; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  // ---- inverse RoPE on output dims [V-R, V) = [448, 512), then store
  if (rg == 3) {
#pragma unroll
    for (int j = 8; j < 16; ++j) {
      const float2 cs = sh.rope[4 * (j - 8) + t4];
      float x0 = om[j][0], x1 = om[j][1];
      om[j][0] = x0 * cs.x + x1 * cs.y;
      om[j][1] = -x0 * cs.y + x1 * cs.x;
      x0 = om[j][2];
      x1 = om[j][3];
      om[j][2] = x0 * cs.x + x1 * cs.y;
      om[j][3] = -x0 * cs.y + x1 * cs.x;
    }
  }
  __nv_bfloat16* o0 = out + ((int64_t)q * kTcH + head0 + g) * kTcV + rg * 128 + 2 * t4;
  __nv_bfloat16* o1 = o0 + 8 * kTcV;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    *reinterpret_cast<uint32_t*>(o0 + 8 * j) = pack_bf16x2(om[j][0], om[j][1]);
    *reinterpret_cast<uint32_t*>(o1 + 8 * j) = pack_bf16x2(om[j][2], om[j][3]);
  }
  if (lse_out && rg == 0 && t4 == 0) {
    lse_out[(int64_t)q * kTcH + head0 + g] = lse_m[0] * kLn2;
    lse_out[(int64_t)q * kTcH + head0 + g + 8] = lse_m[1] * kLn2;
  }
}

// ---------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ float ld1(const T* p, int64_t i);
template <>
__device__ __forceinline__ float ld1<float>(const float* p, int64_t i) { return p[i]; }
template <>
__device__ __forceinline__ float ld1<__nv_bfloat16>(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st1(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st1(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}

constexpr int kSimtMaxVPerLane = 16;  // V <= 512

template <typename T>
__global__ void __launch_bounds__(256) attn_simt_kernel(DevCfg c, DevBatch b, Workspace ws,
                                                        const int* __restrict__ topk_idx,
                                                        const int* __restrict__ topk_cnt,
                                                        T* __restrict__ out,
                                                        float* __restrict__ lse_out) {
  extern __shared__ float sbuf[];  // [warps][V]
  const int q = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  const QueryPlan p = attn_plan(c, b, q, topk_cnt, ws.status, threadIdx.x == 0);
  const int bi = q / b.S;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int V = c.V, D = c.D, R = c.R;
  float* ob = sbuf + warp * V;
  const T* qbase = static_cast<const T*>(b.q) + (int64_t)q * c.H * D;
  for (int h = warp; h < c.H; h += nw) {
    float om[kSimtMaxVPerLane];
    for (int k = 0; k < kSimtMaxVPerLane; ++k) om[k] = 0.f;
    float lse_m = -INFINITY;
    if (!(p.flags & kPlanBad)) {
      const int ns[3] = {p.nwin, p.cnt, p.vis2};
      for (int sid = 0; sid < 3; ++sid) {
        float m = -INFINITY, l = 0.f, oa[kSimtMaxVPerLane];
        for (int k = 0; k < kSimtMaxVPerLane; ++k) oa[k] = 0.f;
        for (int i = 0; i < ns[sid]; ++i) {
          int64_t gr;
          const T* base;
          int64_t stride, rows;
          bool ok = true;
          if (sid == 0) {
            gr = raw_row(b, bi, p.pos - p.nwin + 1 + i);
            base = static_cast<const T*>(b.raw); stride = b.raw_stride; rows = b.raw_rows;
          } else if (sid == 1) {
            const int j = topk_idx[(int64_t)q * c.K + i];
            ok = j >= 0 && j < p.vis;
            gr = cmp_row(b, bi, j);
            base = static_cast<const T*>(b.cmp); stride = b.cmp_stride; rows = b.cmp_rows;
          } else {
            gr = hca_row(b, bi, i);
            base = static_cast<const T*>(b.hca); stride = b.hca_stride; rows = b.hca_rows;
          }
          ok = ok && gr >= 0 && gr < rows;
          if (!ok) {
            if (lane == 0 && h == warp) set_status(ws.status, kStatusBadIndex);
            continue;
          }
          const T* row = base + gr * stride;
          float dot = 0.f;
          for (int d = lane; d < D; d += 32)
            dot = fmaf(ld1(qbase, (int64_t)h * D + d), ld1(row, d), dot);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
          const float s = dot * c.scale;
          const float mn = fmaxf(m, s);
          const float al = expf(m - mn);
          const float pe = expf(s - mn);
          l = l * al + pe;
          for (int k = 0; k < kSimtMaxVPerLane; ++k) {
            const int v = lane + 32 * k;
            if (v < V) oa[k] = oa[k] * al + pe * ld1(row, v);
          }
          m = mn;
        }
        if (l > 0.f) {
          const float lse_s = m + logf(l);
          const float nl = fmaxf(lse_m, lse_s);
          const float wa = expf(lse_m - nl), wb = expf(lse_s - nl);
          const float tot = wa + wb;
          for (int k = 0; k < kSimtMaxVPerLane; ++k) om[k] = (om[k] * wa + oa[k] / l * wb) / tot;
          lse_m = nl + logf(tot);
        }
      }
    }
    for (int k = 0; k < kSimtMaxVPerLane; ++k) {
      const int v = lane + 32 * k;
      if (v < V) ob[v] = om[k];
    }
    __syncwarp();
    if (!(p.flags & kPlanBad)) {
      for (int i = lane; i < R / 2; i += 32) {
        const double ang = (double)p.pos * pow((double)c.rope_base, -2.0 * (double)i / (double)R);
        double sn, cs;
        sincos(ang, &sn, &cs);
        const float x0 = ob[V - R + 2 * i], x1 = ob[V - R + 2 * i + 1];
        ob[V - R + 2 * i] = x0 * (float)cs + x1 * (float)sn;
        ob[V - R + 2 * i + 1] = -x0 * (float)sn + x1 * (float)cs;
      }
    }
    __syncwarp();
    T* orow = out + ((int64_t)q * c.H + h) * V;
    for (int v = lane; v < V; v += 32) st1(orow, v, ob[v]);
    if (lse_out && lane == 0) lse_out[(int64_t)q * c.H + h] = lse_m;
    __syncwarp();
  }
}

}  // namespace

// Attention kernel for the tensor-core shape: the tcgen05 tile kernel +
// merge by default (measured faster); CSA_ATTN=mma selects the warp-MMA
// kernel.
int attention_impl() {
  static const int impl = [] {
    const char* e = getenv("CSA_ATTN");
    return (e && strcmp(e, "mma") == 0) ? kAttnMma : kAttnTc5;
  }();
  return impl;
}

int launch_attention(const DevCfg& c, const DevBatch& b, const Workspace& ws, const int* topk_idx,
                     const int* topk_cnt, void* out, float* lse_out, int num_sms,
                     cudaStream_t st, bool pdl) {
  (void)num_sms;
  const int T = b.B * b.S;
  if (T == 0) return 0;
  if (tensor_core_shape(c)) {
    static PerDeviceOnce attr;
    if (const cudaError_t e = attr.run([] {
          return allow_max_dynamic_smem(attn_tc_kernel);
        }))
      return launch_fail("cudaFuncSetAttribute(attn_tc_kernel)", e);
    return launch_kernel(attn_tc_kernel, dim3(T * 2), dim3(kAttnThreads), kAttnSmem, st, pdl, c, b,
                         ws, topk_idx, topk_cnt, static_cast<__nv_bfloat16*>(out), lse_out);
  }
  const int threads = 256;
  const int smem = (threads / 32) * c.V * 4;
  if (c.dtype == CSA_DTYPE_BF16)
    return launch_kernel(attn_simt_kernel<__nv_bfloat16>, dim3(T), dim3(threads), smem, st, pdl, c,
                         b, ws, topk_idx, topk_cnt, static_cast<__nv_bfloat16*>(out), lse_out);
  return launch_kernel(attn_simt_kernel<float>, dim3(T), dim3(threads), smem, st, pdl, c, b, ws,
                       topk_idx, topk_cnt, static_cast<float*>(out), lse_out);
}

}  // namespace csa
