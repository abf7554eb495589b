// Work planning and split merging for the partial kernel.
//
// mla_plan_kernel      counts the 64-token tiles of every work unit
//                      (request, shard, 64-row query group), forms their
//                      exclusive prefix and picks the tiles per persistent CTA.
// mla_merge_kernel     writes every unit the partial kernel did not write
//                      itself: units with no tokens (o = 0, lse = -inf) and
//                      units split across CTAs, whose pieces it merges by
//                      their LSEs -- the same reweighting that merges shards
//                      ("Decode Context Parallelism", section 4.1).
#include <math_constants.h>

#include "common.cuh"

namespace mla {

__global__ void __launch_bounds__(1024) mla_plan_kernel(ProblemDesc pd, WsHeader* hdr, int* prefix,
                                                        int grid, int min_tiles) {
  __shared__ int part[1024];
  const int U = pd.B * pd.n_out * pd.G;
  const int tid = threadIdx.x;
  const int per_thread = ceil_div(U, 1024);
  const int u0 = tid * per_thread, u1 = min(U, u0 + per_thread);
  int sum = 0;
  for (int u = u0; u < u1; ++u) sum += make_unit(pd, u).tiles;
  part[tid] = sum;
  __syncthreads();
  // inclusive Hillis-Steele scan of the 1024 partial sums
  for (int off = 1; off < 1024; off <<= 1) {
    int v = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int run = part[tid] - sum;  // exclusive
  for (int u = u0; u < u1; ++u) {
    prefix[u] = run;
    run += make_unit(pd, u).tiles;
  }
  if (tid == 1023) {
    const int W = part[1023];
    prefix[U] = W;
    hdr->err = 0;
    hdr->total_tiles = W;
    hdr->per_cta = max(min_tiles, ceil_div(W, grid));
    hdr->grid = grid;
    hdr->num_units = U;
  }
}

__global__ void __launch_bounds__(256) mla_merge_kernel(ProblemDesc pd, const WsHeader* hdr,
                                                        const int* prefix, const float* ws_o,
                                                        const float* ws_lse, float* out_partial,
                                                        float* lse_partial) {
  const int u = blockIdx.x;
  const Unit x = make_unit(pd, u);
  const int us = prefix[u], ue = prefix[u + 1];
  const size_t row0 = ((size_t)x.so * pd.B + x.b) * pd.R + (size_t)x.g * kRows;
  float* dst_o = out_partial + row0 * kDv;
  float* dst_lse = lse_partial + row0;
  const int nvec = x.rows * (kDv / 4);
  if (us == ue) {  // the shard holds no token of this request
    for (int e = threadIdx.x; e < nvec; e += blockDim.x)
      reinterpret_cast<float4*>(dst_o)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = threadIdx.x; r < x.rows; r += blockDim.x) dst_lse[r] = -CUDART_INF_F;
    return;
  }
  const int per = hdr->per_cta;
  const int c0 = us / per, c1 = (ue - 1) / per;
  if (c0 == c1) return;  // written directly by the partial kernel
  auto slot_of = [&](int c) -> size_t {
    return (c == c0 && us > c0 * per) ? 2 * (size_t)c + 1 : 2 * (size_t)c;
  };
  for (int e = threadIdx.x; e < nvec; e += blockDim.x) {
    const int r = e / (kDv / 4), v = e % (kDv / 4);
    float M = -CUDART_INF_F;
    for (int c = c0; c <= c1; ++c) M = fmaxf(M, ws_lse[slot_of(c) * kRows + r]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (M > -CUDART_INF_F) {
      for (int c = c0; c <= c1; ++c) {
        const size_t sl = slot_of(c);
        const float w = __expf(ws_lse[sl * kRows + r] - M);
        const float4 o = reinterpret_cast<const float4*>(ws_o + (sl * kRows + r) * kDv)[v];
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
        wsum += w;
      }
      const float inv = 1.0f / wsum;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
    reinterpret_cast<float4*>(dst_o + (size_t)r * kDv)[v] = acc;
    if (v == 0) dst_lse[r] = (M > -CUDART_INF_F) ? M + __logf(wsum) : -CUDART_INF_F;
  }
}

cudaError_t launch_plan(const ProblemDesc& pd, WsHeader* hdr, int* prefix, int grid,
                        int min_tiles, cudaStream_t stream) {
  mla_plan_kernel<<<1, 1024, 0, stream>>>(pd, hdr, prefix, grid, min_tiles);
  return cudaGetLastError();
}

cudaError_t launch_merge(const ProblemDesc& pd, const WsHeader* hdr, const int* prefix,
                         const float* ws_o, const float* ws_lse, float* out_partial,
                         float* lse_partial, int num_units, cudaStream_t stream) {
  mla_merge_kernel<<<num_units, 256, 0, stream>>>(pd, hdr, prefix, ws_o, ws_lse, out_partial,
                                                  lse_partial);
  return cudaGetLastError();
}

}  // namespace mla
