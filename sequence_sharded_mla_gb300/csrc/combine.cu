// LSE combine of shard partials ("Decode Context Parallelism", section 4.1:
// each shard's partial output is reweighted by its log-sum-exp and the
// weighted partials are summed into the true output), optionally fused with
// the per-head value up-projection W_UV ("Kimi K3 in vLLM: Specialized CuTe
// DSL Decode on NVIDIA GB300", section 1: a fused kernel combines the partial
// results with v-proj).
//
//   M = max_k lse_k,  w_k = exp(lse_k - M),  lse = M + ln sum_k w_k
//   out = sum_k w_k o_k / sum_k w_k                      -> bf16 [rows, 512]
//   y   = out . W_UV[h]   (fp32 out, bf16 weights)       -> bf16 [rows, 128]
//
// The k run over the "pieces" of a row: its N shard partials
// (mla_shard_combine), or, inside a whole decode step, every piece of every
// shard -- a shard's unit computed by one CTA is one piece, a unit split
// across CTAs contributes each CTA's piece.  The merge is associative, so
// merging all pieces of all shards at once equals merging the pieces of each
// shard first and the shards afterwards; no merged per-shard partial is ever
// written back.
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "host_util.h"
#include "merge.cuh"
#include "ptx.cuh"

namespace cg = cooperative_groups;

namespace mla {

namespace {

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Pieces of a row when the N shard partials are stacked shard-major:
// partials [N, rows, 512], lses [N, rows].
struct StackedRows {
  const float* partials;
  const float* lses;
  int num_shards, rows;
  struct Ctx {
    int row, count;
  };
  __device__ Ctx prepare(int row, int /*lane*/) const { return Ctx{row, num_shards}; }
  // Called by every lane of the warp (k may differ per lane, 0 <= k < count).
  __device__ void piece(const Ctx& c, int k, const float*& src, float& lse) const {
    const size_t i = (size_t)k * rows + c.row;
    src = partials + i * kDv;
    lse = __ldg(lses + i);
  }
};

// Pieces of a row of a whole decode step (every shard computed by one
// launch): unit u = (b N + s) G + g of shard s is empty (no piece), written
// whole by one CTA to the step's partial buffer [N, B, R, 512] (one piece),
// or split across CTAs c0..c1 whose pieces are in the workspace slots.
struct StepRows {
  ProblemDesc pd;
  const WsHeader* hdr;
  const int* prefix;
  const float* ws_o;
  const float* ws_lse;
  const float* part;      // [N, B, R, 512]: units written whole
  const float* part_lse;  // [N, B, R]
  struct Ctx {
    int b, rr, r;            // request, row within the request, row within its group
    int count;               // pieces over all shards (warp-uniform)
    int excl, c0, ps, whole; // lane s < N: shard s's first piece index, first CTA,
                             // first work position, whether it is one whole piece
    int per;                 // work positions per CTA (loaded once, not per piece)
  };
  __device__ Ctx prepare(int row, int lane) const {
    Ctx c;
    c.b = row / pd.R;
    c.rr = row - c.b * pd.R;
    const int g = c.rr / kRows;
    c.r = c.rr - g * kRows;
    const int per = hdr->per_cta;
    c.per = per;
    int np = 0;
    c.c0 = 0;
    c.ps = 0;
    c.whole = 0;
    if (lane < pd.num_shards) {
      const int u = (c.b * pd.num_shards + lane) * pd.G + g;
      const Unit x = make_unit(pd, u);
      const int ps = prefix[u], ue = prefix[u + 1];
      const int us = unit_tile_start(prefix, u, hdr->unit_cost);
      // no token to see: an empty shard, or a padding row of a request with
      // fewer query tokens
      if (us < ue && c.r < x.rows) {
        const int c0 = us / per, c1 = (ue - 1) / per;
        c.c0 = c0;
        c.ps = ps;
        c.whole = c0 == c1;
        np = c0 == c1 ? 1 : c1 - c0 + 1;
      }
    }
    int incl = np;
#pragma unroll
    for (int off = 1; off < kMaxShards; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    c.excl = incl - np;
    c.count = __shfl_sync(0xffffffffu, incl, kMaxShards - 1);
    return c;
  }
  __device__ void piece(const Ctx& c, int k, const float*& src, float& lse) const {
    int s = 0;
#pragma unroll
    for (int t = 1; t < kMaxShards; ++t)
      if (t < pd.num_shards && k >= __shfl_sync(0xffffffffu, c.excl, t)) s = t;
    const int ex = __shfl_sync(0xffffffffu, c.excl, s);
    const int c0 = __shfl_sync(0xffffffffu, c.c0, s);
    const int ps = __shfl_sync(0xffffffffu, c.ps, s);
    const int whole = __shfl_sync(0xffffffffu, c.whole, s);
    if (whole) {
      const size_t i = ((size_t)s * pd.B + c.b) * pd.R + c.rr;
      src = part + i * kDv;
      lse = part_lse[i];
    } else {
      // a CTA writes its first piece to slot 0 and its last to slot 1; the
      // unit's first CTA had an earlier piece iff its range starts before
      // the unit's positions
      const int cc = c0 + (k - ex);
      const size_t slot = (cc == c0 && c0 * c.per < ps) ? 2 * (size_t)cc + 1 : 2 * (size_t)cc;
      src = ws_o + (slot * kRows + c.r) * kDv;
      lse = ws_lse[slot * kRows + c.r];
    }
  }
};

// Merges pieces [kbeg, kend) of one row's T pieces (all of them by
// default), a warp at a time, over part of the row: lane `lane` owns the
// float4 columns q0 + lane + 32 v (v < kVec).  The merge is online, batch by
// batch in piece order: a batch's data loads are issued together with its
// LSE loads (the piece addresses need no memory access), the running maximum
// M is raised to the batch's largest LSE and the sums so far are rescaled
// by exp(M_old - M_new).  A typical row is thus two memory round trips (the
// unit lookup, then one batch), and a long request's row -- dozens of
// pieces, every shard's unit split across CTAs -- one round trip per kB
// pieces.  Returns the unnormalised sum acc, M and wsum = sum of
// exp(lse - M) over the warp's pieces (the same value in every lane).
template <int kVec, int kB, class Src>
__device__ __forceinline__ void merge_pieces_ctx(const Src& src, const typename Src::Ctx& ctx,
                                                 int lane, int q0, float4 (&acc)[kVec], float& M,
                                                 float& wsum, int kbeg, int kend) {
#pragma unroll
  for (int v = 0; v < kVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  M = -CUDART_INF_F;
  float ws = 0.f;
  for (int k0 = kbeg; k0 < kend; k0 += 32) {
    const float* p;
    float l;
    src.piece(ctx, min(k0 + lane, kend - 1), p, l);
    if (k0 + lane >= kend) l = -CUDART_INF_F;
    const unsigned long long pa = reinterpret_cast<unsigned long long>(p);
    const int n = min(32, kend - k0);
    for (int j = 0; j < n; j += kB) {
      float4 ob[kB][kVec];
#pragma unroll
      for (int jj = 0; jj < kB; ++jj) {
        const float4* s4 = reinterpret_cast<const float4*>(__shfl_sync(0xffffffffu, pa, j + jj));
        if (j + jj < n) {
#pragma unroll
          for (int v = 0; v < kVec; ++v) ob[jj][v] = s4[q0 + lane + 32 * v];
        }
      }
      float mb = (lane >= j && lane < j + kB) ? l : -CUDART_INF_F;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
      if (mb > M) {
        const float sc = M == -CUDART_INF_F ? 0.f : __expf(M - mb);
#pragma unroll
        for (int v = 0; v < kVec; ++v) {
          acc[v].x *= sc;
          acc[v].y *= sc;
          acc[v].z *= sc;
          acc[v].w *= sc;
        }
        ws *= sc;
        M = mb;
      }
      if (M == -CUDART_INF_F) continue;   // nothing seen yet: every lse so far is -inf
#pragma unroll
      for (int jj = 0; jj < kB; ++jj) {
        const float w = __expf(__shfl_sync(0xffffffffu, l, j + jj) - M);
        if (j + jj < n) {
          ws += w;
#pragma unroll
          for (int v = 0; v < kVec; ++v) {
            acc[v].x = fmaf(w, ob[jj][v].x, acc[v].x);
            acc[v].y = fmaf(w, ob[jj][v].y, acc[v].y);
            acc[v].z = fmaf(w, ob[jj][v].z, acc[v].z);
            acc[v].w = fmaf(w, ob[jj][v].w, acc[v].w);
          }
        }
      }
    }
  }
  wsum = ws;
}


// Warp w handles part w % (4 / kVec) of row w / (4 / kVec) of its block: a
// lane owns kVec float4 of the part's 128 kVec latent dims, so each copy
// instruction of a warp moves 512 contiguous bytes; kB pieces per batch are
// in flight, staged in the warp's slice of dynamic shared memory; at least
// kMinB blocks of 256 threads run per SM.
template <class Src, int kMinB, int kVec, int kB>
__global__ void __launch_bounds__(256, kMinB) mla_combine_kernel(Src src, int rows,
                                                                 uint16_t* __restrict__ out,
                                                                 float* __restrict__ lse_out) {
  constexpr int kWarpsPerRow = 4 / kVec, kRowsPerBlock = 8 / kWarpsPerRow;
  extern __shared__ __align__(16) float4 combine_stage[];   // [8 warps][kB][kVec * 32]
  griddep_wait();                // the partials
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerBlock + warp / kWarpsPerRow, part = warp % kWarpsPerRow;
  if (row >= rows) return;
  float4 acc[kVec];
  float M, wsum;
  const typename Src::Ctx ctx = src.prepare(row, lane);
  merge_pieces_staged<kVec, kB>(src, ctx, lane, 32 * kVec * part,
                                combine_stage + warp * (kB * 32 * kVec), acc, M, wsum);
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(out + (size_t)row * kDv);
#pragma unroll
  for (int v = 0; v < kVec; ++v)
    dst[32 * kVec * part + lane + 32 * v] = make_uint2(pack2(acc[v].x * inv, acc[v].y * inv),
                                                     pack2(acc[v].z * inv, acc[v].w * inv));
  if (lse_out != nullptr && part == 0 && lane == 0)
    lse_out[row] = wsum > 0.f ? M + __logf(wsum) : -CUDART_INF_F;
}

// Fused combine + W_UV, as a cluster of four CTAs that split the 512 latent
// dims.  Cluster (h, rb) handles head h and the query rows (b, i) of block rb
// (kWuvRows of them); CTA q of the cluster merges the dims [128 q, 128 q + 128)
// of those rows (one warp per row, one float4 per lane), multiplies them by
// W_UV[h][128 q .. 128 q + 127][:] (32 KB, staged in shared memory before the
// wait on the preceding kernel), and the four partial projections are summed
// through distributed shared memory, in the fixed order q = 0..3, by CTA q
// for output columns [32 q, 32 q + 32).  Every latent value is merged once
// and W_UV is read once per row block.
constexpr int kWuvRows = 8;            // query rows per cluster (one warp each)
constexpr int kWuvSplit = 4;           // CTAs per cluster
constexpr int kWuvDims = kDv / kWuvSplit;   // 128 latent dims per CTA

// Dynamic shared memory of the W_UV combine kernel.
template <class Src>
struct WuvSmem {
  uint16_t wsm[kWuvDims][kDuv];               // this CTA's 128 rows of W_UV[h] (32 KB)
  float so[kWuvRows][kWuvDims];               // merged latent slice of each row
  float yp[kWuvRows][kDuv];                   // this CTA's partial projection
  float red[8][kWuvRows][kWuvDims];           // per warp and row: sum over its pieces
  float rmax[8][kWuvRows], rsum[8][kWuvRows];
  typename Src::Ctx ctx[kWuvRows][32];        // per row and lane: where its pieces live
  int cnt[kWuvRows];                          // pieces of each row
};

template <class Src>
__global__ void __cluster_dims__(kWuvSplit, 1, 1) __launch_bounds__(256, 2)
    mla_combine_wuv_kernel(Src src, int rows_per_head /* B*q_len */, int H,
                           const uint16_t* __restrict__ w_uv, uint16_t* __restrict__ y,
                           float* __restrict__ lse_out) {
  extern __shared__ __align__(16) uint8_t wuv_smem_raw[];
  WuvSmem<Src>& sm = *reinterpret_cast<WuvSmem<Src>*>(wuv_smem_raw);
  cg::cluster_group cluster = cg::this_cluster();
  const int q = (int)cluster.block_rank();
  const int h = blockIdx.x / kWuvSplit;
  const int rb = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    // W_UV does not depend on the preceding kernel: its copies run while the
    // pieces are located and merged
    const char* wsrc = reinterpret_cast<const char*>(
        w_uv + ((size_t)h * kDv + (size_t)kWuvDims * q) * kDuv);
    const uint32_t wdst = smem_u32(&sm.wsm[0][0]);
    for (int i = tid; i < kWuvDims * kDuv / 8; i += 256) cp_async_16(wdst + 16 * i, wsrc + 16 * i);
    cp_async_commit();
  }
  griddep_wait();                // the partials
  const int bi0 = rb * kWuvRows;
  const int nr = min(kWuvRows, rows_per_head - bi0);
  // where every row's pieces live, one row per warp
  if (warp < nr) {
    sm.ctx[warp][lane] = src.prepare((bi0 + warp) * H + h, lane);
    if (lane == 0) sm.cnt[warp] = sm.ctx[warp][lane].count;
  }
  __syncthreads();
  {
    // The rows' pieces, concatenated in row order, are divided evenly over
    // the 8 warps: a long request's row (dozens of pieces) is merged by
    // several warps at once instead of one round trip after another.
    int total = 0;
    for (int r = 0; r < nr; ++r) total += sm.cnt[r];
    const int lo = (int)((long long)total * warp / 8), hi = (int)((long long)total * (warp + 1) / 8);
    int base = 0;
    for (int r = 0; r < kWuvRows; ++r) {
      const int c = r < nr ? sm.cnt[r] : 0;
      const int k0 = max(lo, base) - base, k1 = min(hi, base + c) - base;
      float M = -CUDART_INF_F, wsum = 0.f;
      float4 acc[1] = {make_float4(0.f, 0.f, 0.f, 0.f)};
      if (k0 < k1) {
        const typename Src::Ctx ctx = sm.ctx[r][lane];
        merge_pieces_ctx<1, 8>(src, ctx, lane, kWuvDims / 4 * q, acc, M, wsum, k0, k1);
      }
      *reinterpret_cast<float4*>(&sm.red[warp][r][4 * lane]) = acc[0];
      if (lane == 0) {
        sm.rmax[warp][r] = M;
        sm.rsum[warp][r] = wsum;
      }
      base += c;
    }
  }
  __syncthreads();
  {
    // row r's merged slice: the warps' parts brought to the row's largest
    // maximum and added in warp order, normalised
    const int r = warp;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < nr) {
      float M = -CUDART_INF_F;
      for (int w = 0; w < 8; ++w) M = fmaxf(M, sm.rmax[w][r]);
      float ws = 0.f;
      if (M > -CUDART_INF_F) {
        for (int w = 0; w < 8; ++w) {
          const float mp = sm.rmax[w][r];
          if (mp == -CUDART_INF_F) continue;
          const float sc = __expf(mp - M);
          const float4 a = *reinterpret_cast<const float4*>(&sm.red[w][r][4 * lane]);
          v.x = fmaf(sc, a.x, v.x);
          v.y = fmaf(sc, a.y, v.y);
          v.z = fmaf(sc, a.z, v.z);
          v.w = fmaf(sc, a.w, v.w);
          ws = fmaf(sc, sm.rsum[w][r], ws);
        }
      }
      const float inv = ws > 0.f ? 1.0f / ws : 0.f;
      v = make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
      if (lse_out != nullptr && q == 0 && lane == 0)
        lse_out[(bi0 + r) * H + h] = ws > 0.f ? M + __logf(ws) : -CUDART_INF_F;
    }
    *reinterpret_cast<float4*>(&sm.so[r][4 * lane]) = v;
  }
  cp_async_wait_all();           // this thread's W_UV copies
  __syncthreads();
  {
    // thread (rh, c): output column c, rows 4 rh .. 4 rh + 3
    const int c = tid & (kDuv - 1), rh = tid >> 7;
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int d = 0; d < kWuvDims; ++d) {
      const float w = __uint_as_float(((uint32_t)sm.wsm[d][c]) << 16);
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = fmaf(sm.so[4 * rh + r][d], w, a[r]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) sm.yp[4 * rh + r][c] = a[r];
  }
  cluster.sync();                // every CTA's partial projection is complete
  {
    // CTA q finalises columns [32 q, 32 q + 32) of the block's rows
    const int r = tid >> 5, c = 32 * q + lane;
    if (r < nr) {
      float v = 0.f;
#pragma unroll
      for (int qq = 0; qq < kWuvSplit; ++qq) {
        const float* peer = cluster.map_shared_rank(&sm.yp[0][0], qq);
        v += peer[r * kDuv + c];
      }
      __nv_bfloat16 b = __float2bfloat16_rn(v);
      y[((size_t)(bi0 + r) * H + h) * kDuv + c] = *reinterpret_cast<uint16_t*>(&b);
    }
  }
  cluster.sync();                // peers' shared memory stays alive until read
}

// The combine is latency-bound.  Many rows (with few pieces each, e.g. a
// verify batch of 9,216 rows) want many rows in flight per SM; fewer rows,
// where long requests bring dozens of pieces per row, want many pieces of
// one row in flight.
constexpr int kManyRows = 4096;
// Pieces per staged batch.  Fewer rows: four warps per row (one float4 per
// lane), 16 pieces in flight per warp, 8 x 16 x 512 B = 64 KB per block,
// three blocks per SM.  Many rows: one warp per row (four float4 per lane,
// all 512 dims), 3 pieces in flight, 8 x 3 x 2 KB = 48 KB: eight rows per
// block, half the blocks of two warps per row, four blocks per SM.
constexpr int kFewB = 16, kManyB = 3;

template <class Src, int kMinB, int kVec, int kB>
cudaError_t launch_combine_shape(const Src& src, int rows, uint16_t* out, float* lse_out,
                                 cudaStream_t stream) {
  constexpr int kRowsPerBlock = 2 * kVec;
  constexpr int smem = 8 * kB * 32 * kVec * (int)sizeof(float4);
  const cudaError_t e = host::ensure_dynamic_smem(
      reinterpret_cast<const void*>(&mla_combine_kernel<Src, kMinB, kVec, kB>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ceil_div(rows, kRowsPerBlock));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_combine_kernel<Src, kMinB, kVec, kB>, src, rows, out, lse_out);
}

template <class Src>
cudaError_t launch_combine_impl(const Src& src, int rows, uint16_t* out, float* lse_out,
                                cudaStream_t stream) {
  if (rows >= kManyRows) return launch_combine_shape<Src, 4, 4, kManyB>(src, rows, out, lse_out, stream);
  return launch_combine_shape<Src, 4, 1, kFewB>(src, rows, out, lse_out, stream);
}

template <class Src>
cudaError_t launch_combine_wuv_impl(const Src& src, int rows_per_head, int H,
                                    const uint16_t* w_uv, uint16_t* y, float* lse_out,
                                    cudaStream_t stream) {
  const int smem = (int)sizeof(WuvSmem<Src>);
  const cudaError_t e = host::ensure_dynamic_smem(
      reinterpret_cast<const void*>(&mla_combine_wuv_kernel<Src>), smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(H * kWuvSplit, ceil_div(rows_per_head, kWuvRows));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_combine_wuv_kernel<Src>, src, rows_per_head, H, w_uv, y,
                            lse_out);
}

}  // namespace

cudaError_t launch_combine(const float* partials, const float* lses, int num_shards, int rows,
                           uint16_t* out, float* lse_out, cudaStream_t stream) {
  return launch_combine_impl(StackedRows{partials, lses, num_shards, rows}, rows, out, lse_out,
                             stream);
}

cudaError_t launch_combine_wuv(const float* partials, const float* lses, int num_shards,
                               int rows_per_head, int H, const uint16_t* w_uv, uint16_t* y,
                               float* lse_out, cudaStream_t stream) {
  return launch_combine_wuv_impl(StackedRows{partials, lses, num_shards, rows_per_head * H},
                                 rows_per_head, H, w_uv, y, lse_out, stream);
}

cudaError_t launch_step_combine(const ProblemDesc& pd, const WsHeader* hdr, const int* prefix,
                                const float* ws_o, const float* ws_lse, const float* part,
                                const float* part_lse, const uint16_t* w_uv, uint16_t* out,
                                float* lse_out, cudaStream_t stream) {
  const StepRows src{pd, hdr, prefix, ws_o, ws_lse, part, part_lse};
  if (w_uv == nullptr) return launch_combine_impl(src, pd.B * pd.R, out, lse_out, stream);
  return launch_combine_wuv_impl(src, pd.B * pd.q_len, pd.H, w_uv, out, lse_out, stream);
}

}  // namespace mla
