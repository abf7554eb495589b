// The W_UV up-projection of the combined latent output on the tensor cores,
// for batches with many query rows per head.
//
// "Kimi K3 in vLLM: Specialized CuTe DSL Decode..." (section 1) fuses the
// v-projection with the combine: y[b,i,h,:] = o[b,i,h,:] . W_UV[h] (512 -> 128).
// The fused combine kernel (combine.cu) does this on the CUDA cores, which is
// right for a few rows per head.  With 64 or more rows per head (verify steps
// with several query tokens, large batches) the projection is one GEMM per
// head, Y_h [rows, 128] = O_h [rows, 512] . W_UV[h] [512, 128], and runs here
// on tcgen05 after the combine has written the normalised O in bf16:
//
//   CTA (row block rb, head h): M = 128 rows (b, i) of head h, N = 128,
//   K = 512 in eight 64-wide chunks through a four-stage ring:
//     A (O rows, K-major)   one TMA box of 128 rows x 64 dims (16 KB) per chunk,
//                           from the view (dim, head, row) of O [rows, H, 512]
//     B (W_UV[h], N-major)  two TMA boxes of 64 k x 64 n (8 KB each) per chunk
//   warp 0 loads, warp 1 issues the MMAs (M128 N128 K16, fp32 accumulator in
//   128 TMEM columns), warps 2..5 (one TMEM lane quadrant each) store the
//   rows' 128 outputs as bf16.
//
// The rows' O is rounded to bf16 before the product, as an unfused projection
// of the bf16 attention output would be.
#include <cuda_bf16.h>

#include "common.cuh"
#include "host_util.h"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kGThreads = 192;
constexpr int kGRows = 128;                  // M: rows of one head per CTA
constexpr int kGN = kDuv;                    // 128 outputs per row
constexpr int kGKChunk = 64;                 // K per stage
constexpr int kGChunks = kDv / kGKChunk;     // 8
constexpr int kGStages = 4;
constexpr int kGABytes = kGRows * kGKChunk * 2;     // 16384
constexpr int kGBHalf = kGKChunk * 64 * 2;          // 8192: 64 k x 64 n
constexpr int kGBBytes = 2 * kGBHalf;               // 16384
constexpr int kGStageBytes = kGABytes + kGBBytes;   // 32768
constexpr int kGSmemBytes = kGStages * kGStageBytes + 1024 + 1024;
constexpr uint32_t kGTmemCols = 128;

struct GMisc {
  uint64_t full[kGStages], empty[kGStages];
  uint64_t done, drain;
  uint32_t tmem_base;
  int abort;
};

}  // namespace

__global__ void __launch_bounds__(kGThreads, 1)
    mla_wuv_gemm_kernel(const __grid_constant__ CUtensorMap tm_o,
                        const __grid_constant__ CUtensorMap tm_w, uint16_t* __restrict__ y,
                        int rows_per_head, int H, unsigned* err, unsigned long long timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  GMisc* misc = reinterpret_cast<GMisc*>(smem + kGStages * kGStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rb = blockIdx.x, h = blockIdx.y;
  const int row0 = rb * kGRows;
  const uint32_t s0 = smem_u32(smem);
  volatile int* abort_flag = &misc->abort;
  auto fail = [&]() {
    atomicOr(err, kErrTimeout);
    *(volatile int*)&misc->abort = 1;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(smem_u32(&misc->full[s]), 1);
      mbar_init(smem_u32(&misc->empty[s]), 1);
    }
    mbar_init(smem_u32(&misc->done), 1);
    mbar_init(smem_u32(&misc->drain), 1);
    misc->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc->tmem_base), kGTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc->tmem_base;
  int armed[kGStages] = {-1, -1, -1, -1};   // producer: last armed use of each stage

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // W_UV does not depend on the preceding kernel: the first stages' B
    // halves go out before the wait for the combine's O.
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tm_o);
      tma_prefetch_desc(&tm_w);
    }
    for (int c = 0; c < kGChunks && ok; ++c) {
      const int s = c % kGStages;
      const uint32_t st = s0 + s * kGStageBytes;
      if (c >= kGStages) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->empty[s]), ((c / kGStages) - 1) & 1,
                                               timeout_ns, abort_flag));
        if (!ok) break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(smem_u32(&misc->full[s]), kGStageBytes);
        armed[s] = c / kGStages;
        // B: k rows 64c .. 64c + 63 of W_UV[h], n halves 0..63 and 64..127
        tma_load_3d(st + kGABytes, &tm_w, smem_u32(&misc->full[s]), 0, kGKChunk * c, h);
        tma_load_3d(st + kGABytes + kGBHalf, &tm_w, smem_u32(&misc->full[s]), 64, kGKChunk * c, h);
        if (c == 0) griddep_wait();     // O is the preceding kernel's output
        // A: dims 64c .. 64c + 63 of rows row0 .. row0 + 127 of head h
        tma_load_3d(st, &tm_o, smem_u32(&misc->full[s]), kGKChunk * c, h, row0);
      }
      __syncwarp();
    }
    if (!ok && lane == 0) fail();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    const uint32_t idesc = idesc_bf16_f32(kGRows, kGN, false, true);
    bool ok = true;
    for (int c = 0; c < kGChunks && ok; ++c) {
      const int s = c % kGStages;
      const uint32_t st = s0 + s * kGStageBytes;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->full[s]), (c / kGStages) & 1,
                                             timeout_ns, abort_flag));
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kGKChunk / 16; ++kk) {
          // A: K-major rows of 128 bytes, 8-row groups 1024 bytes apart
          const uint64_t a = sw128_desc(st + 32 * kk, 16, 1024);
          // B: N-major; the two 64-wide n halves 8 KB apart, 8-k groups
          // 1024 bytes apart, 16 k rows per K16 step
          const uint64_t b = sw128_desc(st + kGABytes + 2048 * kk, kGBHalf, 1024);
          mma_bf16_ss(tmem, a, b, idesc, (c > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&misc->empty[s]));
        if (c == kGChunks - 1) mma_commit(smem_u32(&misc->done));
      }
      __syncwarp();
    }
    if (!ok && lane == 0) fail();
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int r = 32 * quad + lane;
    const bool ok =
        __all_sync(0xffffffffu, mbar_wait(smem_u32(&misc->done), 0, timeout_ns, abort_flag));
    if (!ok) {
      if (lane == 0) fail();
    } else {
      tc_fence_after();
      const int bi = row0 + r;
      uint4* dst = reinterpret_cast<uint4*>(y + ((size_t)bi * H + h) * kGN);
#pragma unroll 1
      for (int c0 = 0; c0 < kGN; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + c0, v);
        tmem_wait_ld();
        if (bi < rows_per_head) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            uint32_t w[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              __nv_bfloat162 p = __floats2bfloat162_rn(__uint_as_float(v[8 * e + 2 * t]),
                                                       __uint_as_float(v[8 * e + 2 * t + 1]));
              w[t] = *reinterpret_cast<uint32_t*>(&p);
            }
            dst[c0 / 8 + e] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // after a failure, the MMAs and copies in flight land before TMEM is
    // freed and the CTA exits
    int never = 0;
    if (warp == 1 && lane == 0) {
      mma_commit(smem_u32(&misc->drain));
      mbar_wait(smem_u32(&misc->drain), 0, kDrainNs, &never);
    }
    if (warp == 0 && lane == 0)
      for (int s = 0; s < kGStages; ++s)
        if (armed[s] >= 0) mbar_wait(smem_u32(&misc->full[s]), armed[s] & 1, kDrainNs, &never);
    tc_fence_before();
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kGTmemCols);
  }
}

cudaError_t launch_wuv_gemm(const uint16_t* o, const uint16_t* w_uv, uint16_t* y,
                            int rows_per_head, int H, unsigned* err,
                            unsigned long long timeout_ns, cudaStream_t stream) {
  host::EncodeTiledFn encode = host::encode_fn();
  if (encode == nullptr) return cudaErrorInitializationError;
  CUtensorMap tm_o, tm_w;
  cuuint32_t es[3] = {1, 1, 1};
  {
    // O [rows, H, 512] bf16 as (dim, head, row)
    cuuint64_t dims[3] = {(cuuint64_t)kDv, (cuuint64_t)H, (cuuint64_t)rows_per_head};
    cuuint64_t strides[2] = {(cuuint64_t)kDv * 2, (cuuint64_t)H * kDv * 2};
    cuuint32_t box[3] = {(cuuint32_t)kGKChunk, 1, (cuuint32_t)kGRows};
    if (encode(&tm_o, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(o), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // W_UV [H, 512, 128] bf16 as (n, k, head)
    cuuint64_t dims[3] = {(cuuint64_t)kGN, (cuuint64_t)kDv, (cuuint64_t)H};
    cuuint64_t strides[2] = {(cuuint64_t)kGN * 2, (cuuint64_t)kDv * kGN * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kGKChunk, 1};
    if (encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(w_uv), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  const cudaError_t e = host::ensure_dynamic_smem(
      reinterpret_cast<const void*>(&mla_wuv_gemm_kernel), kGSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ceil_div(rows_per_head, kGRows), H);
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = kGSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr = pdl_attribute();
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mla_wuv_gemm_kernel, tm_o, tm_w, y, rows_per_head, H, err,
                            timeout_ns);
}

}  // namespace mla
