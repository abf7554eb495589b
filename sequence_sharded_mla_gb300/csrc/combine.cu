// LSE combine of shard partials ("Decode Context Parallelism", section 4.1:
// each shard's partial output is reweighted by its log-sum-exp and the
// weighted partials are summed into the true output), optionally fused with
// the per-head value up-projection W_UV ("Kimi K3 in vLLM: Specialized CuTe
// DSL Decode on NVIDIA GB300", section 1: a fused kernel combines the partial
// results with v-proj).
//
//   M = max_s lse_s,  w_s = exp(lse_s - M),  lse = M + ln sum_s w_s
//   out = sum_s w_s o_s / sum_s w_s                      -> bf16 [rows, 512]
//   y   = out . W_UV[h]   (fp32 out, bf16 weights)       -> bf16 [rows, 128]
#include <cuda_bf16.h>
#include <math_constants.h>

#include "common.cuh"
#include "ptx.cuh"

namespace mla {

namespace {

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace

// Merges one row of the N shard partials by their LSEs into acc (unscaled)
// and returns M = max lse and wsum = sum of exp(lse - M).  Each lane owns 16
// of the 512 dims (four float4 at dims 4*lane + 128*k).  The rows of up to
// four shards and all the LSEs are loaded together, before the weights are
// known, so their latencies overlap; the sum runs over s = 0..N-1 in order.
__device__ __forceinline__ void merge_row(const float* __restrict__ partials,
                                          const float* __restrict__ lses, int num_shards,
                                          int rows, int row, int lane, float4 (&acc)[4], float& M,
                                          float& wsum) {
  float4 ob[4][4];
  auto load4 = [&](int s0) {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (s0 + j < num_shards) {
        const float4* src =
            reinterpret_cast<const float4*>(partials + ((size_t)(s0 + j) * rows + row) * kDv);
#pragma unroll
        for (int k = 0; k < 4; ++k) ob[j][k] = __ldg(src + lane + 32 * k);
      }
  };
  load4(0);
  float l[kMaxShards];
  M = -CUDART_INF_F;
#pragma unroll
  for (int s = 0; s < kMaxShards; ++s) {
    l[s] = s < num_shards ? __ldg(lses + (size_t)s * rows + row) : -CUDART_INF_F;
    M = fmaxf(M, l[s]);
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  wsum = 0.f;
  if (M == -CUDART_INF_F) return;
#pragma unroll
  for (int s0 = 0; s0 < kMaxShards; s0 += 4) {
    if (s0 >= num_shards) break;
    if (s0 > 0) load4(s0);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      if (s0 + j < num_shards) {
        const float w = __expf(l[s0 + j] - M);
        wsum += w;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[k].x += w * ob[j][k].x;
          acc[k].y += w * ob[j][k].y;
          acc[k].z += w * ob[j][k].z;
          acc[k].w += w * ob[j][k].w;
        }
      }
    }
  }
}

// One warp per query row; each lane owns 16 of the 512 latent dims
// (four float4 at dims 4*lane + 128*k), so every load instruction of the warp
// reads 512 contiguous bytes.
__global__ void __launch_bounds__(256) mla_combine_kernel(const float* __restrict__ partials,
                                                          const float* __restrict__ lses,
                                                          int num_shards, int rows,
                                                          uint16_t* __restrict__ out,
                                                          float* __restrict__ lse_out) {
  griddep_wait();                // the partials
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float4 acc[4];
  float M, wsum;
  merge_row(partials, lses, num_shards, rows, row, lane, acc, M, wsum);
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  uint2* dst = reinterpret_cast<uint2*>(out + (size_t)row * kDv);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    dst[lane + 32 * k] = make_uint2(pack2(acc[k].x * inv, acc[k].y * inv),
                                    pack2(acc[k].z * inv, acc[k].w * inv));
  if (lse_out != nullptr && lane == 0)
    lse_out[row] = M > -CUDART_INF_F ? M + __logf(wsum) : -CUDART_INF_F;
}

// Fused combine + W_UV.  Block (h, jb) handles head h and output columns
// [16*jb, 16*jb + 16) for every (b, i) row of that head, 8 rows at a time:
// it merges the shard partials of those rows into shared memory (fp32, one
// warp per row), then 256 threads (16 columns x 16 slices; slice s takes the
// latent dims c = s mod 16) accumulate out . W_UV[h][:, col] and reduce the
// slices.  128 / 16 column blocks per head keep 8 x H blocks in flight: at
// small batches the projection is latency-bound, not bandwidth-bound.  The
// block's W_UV columns (512 x 16 bf16) do not depend on the partials, so they
// are staged in shared memory before the wait on the preceding kernel.
constexpr int kWuvRowsPerPass = 8;
constexpr int kWuvCols = 16;                  // output columns per block
constexpr int kWuvSlices = 256 / kWuvCols;    // 16 slices of 32 latent dims

__global__ void __launch_bounds__(256) mla_combine_wuv_kernel(
    const float* __restrict__ partials, const float* __restrict__ lses, int num_shards,
    int rows_per_head_group /* B*q_len */, int H, const uint16_t* __restrict__ w_uv,
    uint16_t* __restrict__ y, float* __restrict__ lse_out) {
  __shared__ float so[kWuvRowsPerPass][kDv];
  __shared__ float red[kWuvSlices][kWuvRowsPerPass][kWuvCols];
  __shared__ __align__(16) uint16_t wsm[kDv][kWuvCols];
  const int h = blockIdx.x, jb = blockIdx.y;
  const int tid = threadIdx.x;
  {
    // 512 rows x 32 bytes: two 16-byte pieces per row
    const uint16_t* wblk = w_uv + (size_t)h * kDv * kDuv + kWuvCols * jb;
    for (int i = tid; i < kDv * 2; i += blockDim.x) {
      const int c = i >> 1, half = i & 1;
      *reinterpret_cast<uint4*>(&wsm[c][8 * half]) =
          __ldg(reinterpret_cast<const uint4*>(wblk + (size_t)c * kDuv + 8 * half));
    }
  }
  griddep_wait();                // the partials
  const int rows = rows_per_head_group * H;
  const int col = tid & (kWuvCols - 1), slice = tid / kWuvCols;
  const int warp = tid >> 5, lane = tid & 31;
  for (int base = 0; base < rows_per_head_group; base += kWuvRowsPerPass) {
    const int nr = min(kWuvRowsPerPass, rows_per_head_group - base);
    // merge: warp w handles row w of this pass
    if (warp < nr) {
      const int row = (base + warp) * H + h;
      float4 acc[4];
      float M, wsum;
      merge_row(partials, lses, num_shards, rows, row, lane, acc, M, wsum);
      const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float4 v = make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
        *reinterpret_cast<float4*>(&so[warp][4 * (lane + 32 * k)]) = v;
      }
      if (lse_out != nullptr && jb == 0 && lane == 0)
        lse_out[row] = M > -CUDART_INF_F ? M + __logf(wsum) : -CUDART_INF_F;
    }
    __syncthreads();
    float acc[kWuvRowsPerPass];
#pragma unroll
    for (int r = 0; r < kWuvRowsPerPass; ++r) acc[r] = 0.f;
#pragma unroll 8
    for (int c = slice; c < kDv; c += kWuvSlices) {
      const float w = __uint_as_float(((uint32_t)wsm[c][col]) << 16);
#pragma unroll
      for (int r = 0; r < kWuvRowsPerPass; ++r) acc[r] += so[r][c] * w;
    }
#pragma unroll
    for (int r = 0; r < kWuvRowsPerPass; ++r) red[slice][r][col] = acc[r];
    __syncthreads();
    if (tid < nr * kWuvCols) {
      const int r = tid / kWuvCols, c = tid % kWuvCols;
      float v = 0.f;
#pragma unroll
      for (int sl = 0; sl < kWuvSlices; ++sl) v += red[sl][r][c];
      const int row = (base + r) * H + h;
      __nv_bfloat16 b = __float2bfloat16_rn(v);
      y[(size_t)row * kDuv + kWuvCols * jb + c] = *reinterpret_cast<uint16_t*>(&b);
    }
    __syncthreads();
  }
}

cudaError_t launch_combine(const float* partials, const float* lses, int num_shards, int rows,
                           uint16_t* out, float* lse_out, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ceil_div(rows, 8));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_combine_kernel, partials, lses, num_shards, rows, out,
                            lse_out);
}

cudaError_t launch_combine_wuv(const float* partials, const float* lses, int num_shards,
                               int rows_per_head_group, int H, const uint16_t* w_uv, uint16_t* y,
                               float* lse_out, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(H, kDuv / kWuvCols);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_combine_wuv_kernel, partials, lses, num_shards,
                            rows_per_head_group, H, w_uv, y, lse_out);
}

}  // namespace mla
