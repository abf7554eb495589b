// LSE merge of a row's pieces with each batch staged in shared memory.
// Shared by the combine kernels and the merge of split units.
//
// A piece source `Src` provides a context type `Src::Ctx` (with a member
// `count`, the row's pieces) and `piece(ctx, k, src, lse)`, called by every
// lane of a warp with its own k (0 <= k < count), returning the address of
// piece k's row (512 fp32) and its LSE.  The merge is online, batch by batch
// in piece order:
//
//   M = max_k lse_k,  w_k = exp(lse_k - M),  acc = sum_k w_k o_k,  wsum = sum_k w_k
//
// ("Decode Context Parallelism", section 4.1: each partial output is
// reweighted by its log-sum-exp).
#pragma once

#include <math_constants.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

// Lane `lane` owns the float4 columns q0 + lane + 32 v (v < kVec) of the
// row.  Each batch of kB pieces is staged in shared memory by cp.async: the
// lane copies its kVec float4 of every piece of the batch into `stage` (its
// warp's [kB][kVec * 32] float4) and reads back only what it copied, so the
// bytes in flight hold no registers and kB can be several times what the
// register file allows.  Returns the unnormalised sum acc, M and wsum (the
// same M and wsum in every lane).
template <int kVec, int kB, class Src>
__device__ __forceinline__ void merge_pieces_staged(const Src& src, const typename Src::Ctx& ctx,
                                                    int lane, int q0, float4* stage,
                                                    float4 (&acc)[kVec], float& M, float& wsum) {
#pragma unroll
  for (int v = 0; v < kVec; ++v) acc[v] = make_float4(0.f, 0.f, 0.f, 0.f);
  M = -CUDART_INF_F;
  float ws = 0.f;
  const int kend = ctx.count;
  for (int k0 = 0; k0 < kend; k0 += 32) {
    const float* p;
    float l;
    src.piece(ctx, min(k0 + lane, kend - 1), p, l);
    if (k0 + lane >= kend) l = -CUDART_INF_F;
    const unsigned long long pa = reinterpret_cast<unsigned long long>(p);
    const int n = min(32, kend - k0);
    for (int j = 0; j < n; j += kB) {
#pragma unroll
      for (int jj = 0; jj < kB; ++jj) {
        const float4* s4 = reinterpret_cast<const float4*>(__shfl_sync(0xffffffffu, pa, j + jj));
        if (j + jj < n) {
#pragma unroll
          for (int v = 0; v < kVec; ++v)
            cp_async_16(smem_u32(stage + jj * (32 * kVec) + lane + 32 * v), s4 + q0 + lane + 32 * v);
        }
      }
      cp_async_commit();
      float mb = (lane >= j && lane < j + kB) ? l : -CUDART_INF_F;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, off));
      cp_async_wait_all();
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
            const float4 o = stage[jj * (32 * kVec) + lane + 32 * v];
            acc[v].x = fmaf(w, o.x, acc[v].x);
            acc[v].y = fmaf(w, o.y, acc[v].y);
            acc[v].z = fmaf(w, o.z, acc[v].z);
            acc[v].w = fmaf(w, o.w, acc[v].w);
          }
        }
      }
    }
  }
  wsum = ws;
}

}  // namespace mla
