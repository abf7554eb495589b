// Work planning and split merging for the partial kernel.
//
// mla_plan_kernel      counts the 64-token tiles of every work unit
//                      (request, shard, 64-row query group), charges every
//                      unit with tiles unit_cost extra positions for its fixed
//                      costs, forms the exclusive prefix of these work
//                      positions and splits them evenly over the persistent
//                      CTAs (a CTA with many short units gets fewer tiles).
// mla_merge_kernel     writes every unit the partial kernel did not write
//                      itself: units with no tokens (o = 0, lse = -inf) and
//                      units split across CTAs, whose pieces it merges by
//                      their LSEs -- the same reweighting that merges shards
//                      ("Decode Context Parallelism", section 4.1).
#include <math_constants.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

__global__ void __launch_bounds__(1024) mla_plan_kernel(ProblemDesc pd, WsHeader* hdr, int* prefix,
                                                        int grid, int min_tiles,
                                                        int unit_cost) {
  griddep_launch_dependents();   // the partial kernel may start launching
  __shared__ unsigned bad_qlen;
  if (threadIdx.x == 0) bad_qlen = 0;
  __syncthreads();
  if (pd.q_lens != nullptr)
    for (int b = threadIdx.x; b < pd.B; b += 1024)
      if (pd.q_lens[b] < 1 || pd.q_lens[b] > pd.q_len) atomicOr(&bad_qlen, kErrQLens);
  __syncthreads();
  plan_units(pd.B * pd.n_out * pd.G, [&](int u) { return make_unit(pd, u).tiles; }, hdr, prefix,
             grid, min_tiles, unit_cost, bad_qlen);
}

// Block (u, y) handles query rows [4y, 4y + 4) of unit u, one warp per row:
// the warp forms the row's piece weights once (in shared memory), then each
// lane accumulates 16 of the 512 latent dims over the pieces.
constexpr int kMergeRowsPerBlock = 4;
constexpr int kMaxPieces = 512;    // pieces of one unit <= persistent CTAs

__global__ void __launch_bounds__(32 * kMergeRowsPerBlock) mla_merge_kernel(
    ProblemDesc pd, const WsHeader* hdr, const int* prefix, const float* ws_o,
    const float* ws_lse, float* out_partial, float* lse_partial) {
  __shared__ float wts[kMergeRowsPerBlock][kMaxPieces];
  griddep_wait();                // the partial kernel's pieces and outputs
  griddep_launch_dependents();
  const int u = blockIdx.x;
  const Unit x = make_unit(pd, u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * kMergeRowsPerBlock + warp;
  if (r >= x.rows_out) return;
  const int ps = prefix[u], ue = prefix[u + 1];
  const int us = unit_tile_start(prefix, u, hdr->unit_cost);
  const size_t orow = out_row(pd, x, r);
  float4* dst = reinterpret_cast<float4*>(out_partial + orow * kDv);
  const int per = hdr->per_cta;
  const bool split = us < ue && us / per != (ue - 1) / per;
  // rows with no token to see: the shard holds none of the request's
  // positions, or the row is padding of a request with fewer query tokens
  // (a whole unit's padding rows are written by the partial kernel)
  if (us == ue || (split && r >= x.rows)) {
    for (int v = lane; v < kDv / 4; v += 32) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane == 0) lse_partial[orow] = -CUDART_INF_F;
    return;
  }
  const int c0 = us / per, c1 = (ue - 1) / per;
  if (c0 == c1) return;  // written directly by the partial kernel
  const int np = c1 - c0 + 1;
  // a CTA writes its first piece to slot 0 and its last to slot 1; the first
  // CTA of the unit had an earlier piece iff its range starts before the
  // unit's positions (the position before them is another unit's tile)
  auto slot_of = [&](int c) -> size_t {
    return (c == c0 && c0 * per < ps) ? 2 * (size_t)c + 1 : 2 * (size_t)c;
  };
  // the first two pieces' rows are loaded before the weights are known, so
  // their latency overlaps the LSE reduction (most split units have two)
  float4 o0[4], o1[4];
  {
    const float4* s0 = reinterpret_cast<const float4*>(ws_o + (slot_of(c0) * kRows + r) * kDv);
    const float4* s1 = reinterpret_cast<const float4*>(ws_o + (slot_of(c0 + 1) * kRows + r) * kDv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o0[i] = s0[lane + 32 * i];
      o1[i] = s1[lane + 32 * i];
    }
  }
  float M = -CUDART_INF_F;
  for (int k = lane; k < np; k += 32) M = fmaxf(M, ws_lse[slot_of(c0 + k) * kRows + r]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float wsum = 0.f;
  for (int k = lane; k < np; k += 32) {
    const float w = M > -CUDART_INF_F ? __expf(ws_lse[slot_of(c0 + k) * kRows + r] - M) : 0.f;
    wts[warp][k] = w;
    wsum += w;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, off);
  __syncwarp();
  float4 acc[4];
  {
    const float w0 = wts[warp][0], w1 = wts[warp][1];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[i].x = w0 * o0[i].x + w1 * o1[i].x;
      acc[i].y = w0 * o0[i].y + w1 * o1[i].y;
      acc[i].z = w0 * o0[i].z + w1 * o1[i].z;
      acc[i].w = w0 * o0[i].w + w1 * o1[i].w;
    }
  }
  for (int k = 2; k < np; ++k) {
    const float w = wts[warp][k];
    const float4* src = reinterpret_cast<const float4*>(ws_o + (slot_of(c0 + k) * kRows + r) * kDv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float4 o = src[lane + 32 * i];
      acc[i].x += w * o.x;
      acc[i].y += w * o.y;
      acc[i].z += w * o.z;
      acc[i].w += w * o.w;
    }
  }
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    dst[lane + 32 * i] = make_float4(acc[i].x * inv, acc[i].y * inv, acc[i].z * inv, acc[i].w * inv);
  if (lane == 0) lse_partial[orow] = wsum > 0.f ? M + __logf(wsum) : -CUDART_INF_F;
}

cudaError_t launch_plan(const ProblemDesc& pd, WsHeader* hdr, int* prefix, int grid,
                        int min_tiles, int unit_cost, cudaStream_t stream) {
  mla_plan_kernel<<<1, 1024, 0, stream>>>(pd, hdr, prefix, grid, min_tiles, unit_cost);
  return cudaGetLastError();
}

cudaError_t launch_merge(const ProblemDesc& pd, const WsHeader* hdr, const int* prefix,
                         const float* ws_o, const float* ws_lse, float* out_partial,
                         float* lse_partial, int num_units, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_units, kRows / kMergeRowsPerBlock);
  cfg.blockDim = dim3(32 * kMergeRowsPerBlock);
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_merge_kernel, pd, hdr, prefix, ws_o, ws_lse, out_partial,
                            lse_partial);
}

}  // namespace mla
