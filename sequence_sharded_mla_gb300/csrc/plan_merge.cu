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
#include "host_util.h"
#include "merge.cuh"
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

// The pieces of a split unit: CTA c0 + k's piece of the unit, in the
// workspace slot it wrote (a CTA writes its first piece to slot 0 and its
// last to slot 1; the unit's first CTA had an earlier piece iff its range
// starts before the unit's positions).
struct UnitPieces {
  const float* ws_o;
  const float* ws_lse;
  struct Ctx {
    int c0, count, r, first_in_slot1;
  };
  __device__ void piece(const Ctx& c, int k, const float*& src, float& lse) const {
    const size_t cc = (size_t)(c.c0 + k);
    const size_t slot = (k == 0 && c.first_in_slot1) ? 2 * cc + 1 : 2 * cc;
    src = ws_o + (slot * kRows + c.r) * kDv;
    lse = ws_lse[slot * kRows + c.r];
  }
};

// Block (u, y) handles query rows 2y and 2y + 1 of unit u with four warps
// per row, each merging 128 of the 512 latent dims over the unit's pieces
// (kMergeBatch pieces in flight per warp).
constexpr int kMergeRowsPerBlock = 2;
constexpr int kMergeBatch = 12;
constexpr int kMergeSmem = 8 * kMergeBatch * 32 * (int)sizeof(float4);

__global__ void __launch_bounds__(256, 4) mla_merge_kernel(
    ProblemDesc pd, const WsHeader* hdr, const int* prefix, const float* ws_o,
    const float* ws_lse, float* out_partial, float* lse_partial) {
  extern __shared__ __align__(16) float4 merge_stage[];   // [8 warps][kMergeBatch][32]
  griddep_wait();                // the partial kernel's pieces and outputs
  griddep_launch_dependents();
  const int u = blockIdx.x;
  const Unit x = make_unit(pd, u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * kMergeRowsPerBlock + (warp >> 2), part = warp & 3;
  if (r >= x.rows_out) return;
  const int ps = prefix[u], ue = prefix[u + 1];
  const int us = unit_tile_start(prefix, u, hdr->unit_cost);
  const size_t orow = out_row(pd, x, r);
  float4* dst = reinterpret_cast<float4*>(out_partial + orow * kDv) + 32 * part;
  const int per = hdr->per_cta;
  const bool split = us < ue && us / per != (ue - 1) / per;
  // rows with no token to see: the shard holds none of the request's
  // positions, or the row is padding of a request with fewer query tokens
  // (a whole unit's padding rows are written by the partial kernel)
  if (us == ue || (split && r >= x.rows)) {
    dst[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (part == 0 && lane == 0) lse_partial[orow] = -CUDART_INF_F;
    return;
  }
  const int c0 = us / per, c1 = (ue - 1) / per;
  if (c0 == c1) return;  // written directly by the partial kernel
  const UnitPieces src{ws_o, ws_lse};
  const UnitPieces::Ctx ctx{c0, c1 - c0 + 1, r, c0 * per < ps ? 1 : 0};
  float4 acc[1];
  float M, wsum;
  merge_pieces_staged<1, kMergeBatch>(src, ctx, lane, 32 * part,
                                      merge_stage + warp * (kMergeBatch * 32), acc, M, wsum);
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  dst[lane] = make_float4(acc[0].x * inv, acc[0].y * inv, acc[0].z * inv, acc[0].w * inv);
  if (part == 0 && lane == 0) lse_partial[orow] = wsum > 0.f ? M + __logf(wsum) : -CUDART_INF_F;
}

cudaError_t launch_plan(const ProblemDesc& pd, WsHeader* hdr, int* prefix, int grid,
                        int min_tiles, int unit_cost, cudaStream_t stream) {
  mla_plan_kernel<<<1, 1024, 0, stream>>>(pd, hdr, prefix, grid, min_tiles, unit_cost);
  return cudaGetLastError();
}

cudaError_t launch_merge(const ProblemDesc& pd, const WsHeader* hdr, const int* prefix,
                         const float* ws_o, const float* ws_lse, float* out_partial,
                         float* lse_partial, int num_units, cudaStream_t stream) {
  const cudaError_t e =
      host::ensure_dynamic_smem(reinterpret_cast<const void*>(&mla_merge_kernel), kMergeSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_units, kRows / kMergeRowsPerBlock);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = kMergeSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_merge_kernel, pd, hdr, prefix, ws_o, ws_lse, out_partial,
                            lse_partial);
}

}  // namespace mla
