// Host side of the C ABI declared in include/mla_dcp.h: argument checks,
// workspace layout, TMA descriptor encoding and kernel launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "mla_dcp.h"
#include "common.cuh"
#include "host_util.h"

namespace mla {
int partial_smem_bytes();
cudaError_t launch_partial_bf16(const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                                const CUtensorMap& tm_kv_pf, const PartialParams& p, int grid,
                                cudaStream_t stream);
cudaError_t launch_partial_fp8(const CUtensorMap& tm_q, const CUtensorMap& tm_kv,
                               const PartialParams& p, int grid, cudaStream_t stream);
cudaError_t launch_plan(const ProblemDesc& pd, WsHeader* hdr, int* prefix, int grid,
                        int min_tiles, int unit_cost, cudaStream_t stream);
cudaError_t launch_merge(const ProblemDesc& pd, const WsHeader* hdr, const int* prefix,
                         const float* ws_o, const float* ws_lse, float* out_partial,
                         float* lse_partial, int num_units, cudaStream_t stream);
cudaError_t launch_combine(const float* partials, const float* lses, int num_shards, int rows,
                           uint16_t* out, float* lse_out, cudaStream_t stream);
cudaError_t launch_combine_wuv(const float* partials, const float* lses, int num_shards,
                               int rows_per_head_group, int H, const uint16_t* w_uv, uint16_t* y,
                               float* lse_out, cudaStream_t stream);
cudaError_t launch_wuv_gemm(const uint16_t* o, const uint16_t* w_uv, uint16_t* y,
                            int rows_per_head, int H, unsigned* err,
                            unsigned long long timeout_ns, cudaStream_t stream);
cudaError_t launch_step_combine(const ProblemDesc& pd, const WsHeader* hdr, const int* prefix,
                                const float* ws_o, const float* ws_lse, const float* part,
                                const float* part_lse, const uint16_t* w_uv, uint16_t* out,
                                float* lse_out, cudaStream_t stream);
}  // namespace mla

using namespace mla;

namespace {

constexpr int kVersion = 200;  // 0.2.0
constexpr unsigned long long kTimeoutNs = 2000000000ull;  // device waits give up after 2 s
constexpr int kMinTilesPerCta = 4;
// Work positions charged to a unit for its fixed costs (query load, pipeline
// refill without the L2 prefetch, the epilogue's 128 KB of output): about
// three tiles' time (measured: 2, 3, 4 and 5 on the bimodal batch 0.546,
// 0.532, 0.530, 0.530 ms; on the q_len-9 batch 3 is best).
constexpr int kUnitCost = 3;
// The fp8 kernel's fixed cost per piece is far larger in tiles (its tiles
// are half the bytes, and a piece splits its query into two e4m3 terms and
// refills four stages): per CTA, one more piece ended the CTA ≈13.5 µs
// later, about 22 of its tiles.  Measured on the long-tail fp8 batch: 3, 10,
// 16 and 24 gave 0.296, 0.291, 0.293 and 0.295 ms.
constexpr int kUnitCostFp8 = 10;

using host::aligned16;
using host::aligned4;
using host::device_sm_count;
using host::encode_fn;
using host::EncodeTiledFn;

struct WsLayout {
  size_t hdr, prefix, ws_o, ws_lse, total;
};

WsLayout ws_layout(int num_units, int grid) {
  auto up = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  WsLayout w;
  w.hdr = 0;
  w.prefix = up(sizeof(WsHeader));
  w.ws_o = w.prefix + up(sizeof(int) * (size_t)(num_units + 1));
  w.ws_lse = w.ws_o + up(sizeof(float) * (size_t)grid * 2 * kRows * kDv);
  w.total = w.ws_lse + up(sizeof(float) * (size_t)grid * 2 * kRows);
  return w;
}

bool shape_ok(const mla_shape* s) {
  return s != nullptr && s->batch >= 1 && s->q_len >= 1 && s->num_heads >= 1 &&
         (s->causal == 0 || s->causal == 1) && std::isfinite(s->softmax_scale) &&
         s->softmax_scale > 0.f && (long long)s->batch * s->q_len * s->num_heads < (1LL << 30);
}

int units_for(const mla_shape* s, int num_shards, int shard_id) {
  int n_out = shard_id == MLA_ALL_SHARDS ? num_shards : 1;
  int G = ceil_div(s->q_len * s->num_heads, kRows);
  return s->batch * n_out * G;
}

}  // namespace

extern "C" {

int mla_version(void) { return kVersion; }

const char* mla_status_string(mla_status st) {
  switch (st) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_TIMEOUT: return "device wait timed out";
    case MLA_ERR_DEVICE_BOUNDS: return "block-table entry out of range";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_RANGE: return "non-finite query value (fp8 cache)";
  }
  return "unknown status";
}

size_t mla_workspace_size(const mla_shape* shape, int num_shards, int shard_id) {
  if (!shape_ok(shape) || num_shards < 1 || num_shards > kMaxShards) return 0;
  if (shard_id != MLA_ALL_SHARDS && (shard_id < 0 || shard_id >= num_shards)) return 0;
  int grid = std::min(device_sm_count(), 512);
  if (grid <= 0) return 0;
  return ws_layout(units_for(shape, num_shards, shard_id), grid).total;
}

}  // extern "C"

namespace {

// What a partial-attention launch leaves for the kernel that completes it
// (the merge of split pieces, or the combine of a whole decode step).
struct Launched {
  ProblemDesc pd;
  WsHeader* hdr;
  int* prefix;
  float* ws_o;
  float* ws_lse;
  int num_units;
};

// Checks the arguments, encodes the tensor maps and launches the planning
// and partial-attention kernels.  Units that one CTA computes whole are
// written to out_partial / lse_partial; pieces of split units to the
// workspace slots described by *L.
// The DCP rank-major I/O of mla_decode_partial_dcp (rank_heads = 0: none).
struct RankIo {
  int rank_heads;   // H / ranks
  int ranks;
  int batch_total;  // requests in the gathered query buffer
  int batch_first;  // first of them computed by this call
};

mla_status partial_launch(const void* q, const mla_kv_pages* kv, const int32_t* block_table,
                          int max_pages_per_req, const int32_t* seq_lens, const mla_shape* shape,
                          int shard_id, int num_shards, mla_layout layout, float* out_partial,
                          float* lse_partial, void* workspace, size_t workspace_bytes,
                          void* stream, Launched* L, RankIo rio = RankIo{0, 1, 0, 0}) {
  if (!q || !kv || !block_table || !seq_lens || !out_partial || !lse_partial) return MLA_ERR_INVALID;
  if (!shape_ok(shape)) return MLA_ERR_INVALID;
  if (num_shards < 1 || num_shards > kMaxShards) return MLA_ERR_INVALID;
  if (shard_id != MLA_ALL_SHARDS && (shard_id < 0 || shard_id >= num_shards)) return MLA_ERR_INVALID;
  if (layout != MLA_LAYOUT_INTERLEAVED && layout != MLA_LAYOUT_CONTIGUOUS &&
      layout != MLA_LAYOUT_INTERLEAVED_LOCAL && layout != MLA_LAYOUT_CONTIGUOUS_LOCAL)
    return MLA_ERR_INVALID;
  const bool local = layout == MLA_LAYOUT_INTERLEAVED_LOCAL || layout == MLA_LAYOUT_CONTIGUOUS_LOCAL;
  if (local && shard_id == MLA_ALL_SHARDS) return MLA_ERR_INVALID;   // a local cache is one shard's
  if (kv->data == nullptr || kv->num_pages < 1 || max_pages_per_req < 1) return MLA_ERR_INVALID;
  if (kv->page_size != kPage) return MLA_ERR_UNSUPPORTED;
  if (kv->dtype == MLA_KV_BF16) {
    if (kv->scale != nullptr) return MLA_ERR_INVALID;
  } else if (kv->dtype == MLA_KV_FP8_E4M3) {
    if (kv->scale == nullptr || !aligned16(kv->scale)) return MLA_ERR_INVALID;
  } else {
    return MLA_ERR_INVALID;
  }
  if (shape->num_heads % 16 != 0) return MLA_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(kv->data) || !aligned16(out_partial) ||
      !aligned16(lse_partial) || !aligned4(block_table) || !aligned4(seq_lens) ||
      !aligned4(shape->q_lens))
    return MLA_ERR_INVALID;
  if (workspace == nullptr || !aligned16(workspace)) return MLA_ERR_WORKSPACE;
  // one persistent CTA per SM (at most 512: the merge keeps per-piece
  // weights of a unit in shared memory)
  const int grid = std::min(device_sm_count(), 512);
  if (grid <= 0) return MLA_ERR_CUDA;
  const int U = units_for(shape, num_shards, shard_id);
  const WsLayout wl = ws_layout(U, grid);
  if (workspace_bytes < wl.total) return MLA_ERR_WORKSPACE;
  EncodeTiledFn encode = encode_fn();
  if (encode == nullptr) return MLA_ERR_CUDA;

  ProblemDesc pd;
  pd.B = shape->batch;
  pd.q_len = shape->q_len;
  pd.H = shape->num_heads;
  pd.R = shape->q_len * shape->num_heads;
  pd.G = ceil_div(pd.R, kRows);
  pd.num_shards = num_shards;
  pd.shard_first = shard_id == MLA_ALL_SHARDS ? 0 : shard_id;
  pd.n_out = shard_id == MLA_ALL_SHARDS ? num_shards : 1;
  pd.layout = (layout == MLA_LAYOUT_INTERLEAVED || layout == MLA_LAYOUT_INTERLEAVED_LOCAL)
                  ? kInterleaved
                  : kContiguous;
  pd.local = local ? 1 : 0;
  // interleaved shards of a whole-request cache: pages per tile and slots
  // per page (padded when N does not divide 64)
  pd.ppt = 1;
  pd.spp_log2 = 6;
  pd.pad = 0;
  pd.rank_heads = rio.rank_heads;
  pd.q_batch_total = rio.rank_heads ? rio.batch_total : pd.B;
  pd.q_batch_first = rio.rank_heads ? rio.batch_first : 0;
  if (layout == MLA_LAYOUT_INTERLEAVED) {
    if (kPage % num_shards == 0) {
      pd.ppt = num_shards;
      pd.spp_log2 = num_shards == 1 ? 6 : num_shards == 2 ? 5 : num_shards == 4 ? 4 : 3;
    } else {
      pd.pad = 1;
      pd.ppt = num_shards == 3 ? 2 : 4;
      pd.spp_log2 = num_shards == 3 ? 5 : 4;
    }
  }
  pd.causal = shape->causal;
  pd.num_pages = kv->num_pages;
  pd.max_pages = max_pages_per_req;
  pd.scale_log2 = shape->softmax_scale * 1.4426950408889634f;
  pd.block_table = block_table;
  pd.seq_lens = seq_lens;
  pd.q_lens = shape->q_lens;

  // query rows: [B*q_len*H, 576] bf16.  Preferred view [rows][9 chunks][64]
  // read as (64 dims, rows, chunk) so one box lands a 64-row group in the
  // [chunk][row][64] shared-memory layout; fallback: one box per chunk.
  CUtensorMap tm_q, tm_kv, tm_kv_pf;
  int q_one_box = 1;
  // rank-major gathered query [ranks, batch_total, q_len, rank_heads, 576]:
  // rows of one rank's heads of one query position are consecutive, so the
  // kernels load a 64-row group as runs of min(rank_heads, 64) rows
  const cuuint64_t q_rows_rm = (cuuint64_t)rio.ranks * rio.batch_total * shape->q_len * rio.rank_heads;
  const cuuint32_t q_run = (cuuint32_t)std::min(rio.rank_heads, kRows);
  if (rio.rank_heads != 0) {
    q_one_box = 0;
    cuuint64_t d2[2] = {(cuuint64_t)kDqk, q_rows_rm};
    cuuint64_t s2[1] = {(cuuint64_t)kDqk * 2};
    cuuint32_t b2[2] = {64, q_run};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), d2, s2, b2, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_CUDA;
  } else {
    cuuint64_t dims[3] = {64, (cuuint64_t)pd.B * pd.R, (cuuint64_t)kChunks};
    cuuint64_t strides[2] = {(cuuint64_t)kDqk * 2, 128};
    cuuint32_t box[3] = {64, (cuuint32_t)kRows, (cuuint32_t)kChunks};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      q_one_box = 0;
      cuuint64_t d2[2] = {(cuuint64_t)kDqk, (cuuint64_t)pd.B * pd.R};
      cuuint64_t s2[1] = {(cuuint64_t)kDqk * 2};
      cuuint32_t b2[2] = {64, (cuuint32_t)kRows};
      if (encode(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(q), d2, s2, b2, es,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MLA_ERR_CUDA;
    }
  }
  // cache rows, nv = N for interleaved shards (else 1): a tile's 64 slots
  // are nv pages x 64/nv rows, slot a in 8-slot group a/8.  The bf16 view
  // (64 dims, row in group, chunk, group, cache row) with strides
  // (-, 1152 nv, 128, 9216 nv, 1152) starts at cache row page*64 + residue
  // and lands the residue's 64/nv rows of a page in the kernels'
  // shared-memory layouts: all 9 chunks of each 8-slot group in one box
  // (fp8), or three chunks per box, one box per chunk group (bf16).
  // nv pages per tile, 64 / nv slots per page (padded for N not dividing 64)
  const int nv = pd.ppt;
  const bool fp8 = kv->dtype == MLA_KV_FP8_E4M3;
  CUtensorMap tm_q8;
  if (fp8) {
    // query rows for the fp8 kernel, by 8-row groups: view (64 dims, row in
    // group, chunk, row group) with strides (-, 1152, 128, 9216); a box lands
    // a 64-row group as [row group][chunk][row][64], 9216 bytes per row group
    cuuint64_t qd[4] = {64, 8, (cuuint64_t)kChunks,
                        rio.rank_heads ? q_rows_rm / 8 : (cuuint64_t)pd.B * pd.R / 8};
    cuuint64_t qs[3] = {(cuuint64_t)kDqk * 2, 128, (cuuint64_t)kDqk * 2 * 8};
    cuuint32_t qb[4] = {64, 8, (cuuint32_t)kChunks, rio.rank_heads ? q_run / 8 : (cuuint32_t)(kRows / 8)};
    cuuint32_t qe[4] = {1, 1, 1, 1};
    if (encode(&tm_q8, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), qd, qs, qb, qe,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_CUDA;
    // e4m3 codes: the same view with 64-code chunks, strides (-, 576 nv, 64,
    // 4608 nv, 576) and 64-byte swizzling: a box lands a page's residue rows,
    // all nine chunks, in the group-major layout of the fp8 kernel.  No L2
    // promotion: a 576-byte row is 18 whole sectors, and promotion to 128
    // bytes would fetch 640
    if (pd.pad) {
      // N does not divide 64: view (64 codes, row in page, chunk, page) with
      // strides (-, 576, 64, 36864); a box of 8 N rows traversed with stride
      // N lands one 8-slot group (4608 bytes), and rows past the page's end
      // are outside the view and fill zeros
      cuuint64_t pdims[4] = {64, (cuuint64_t)kPage, (cuuint64_t)kChunks,
                             (cuuint64_t)kv->num_pages};
      cuuint64_t pstrides[3] = {(cuuint64_t)kDqk, 64, (cuuint64_t)kDqk * kPage};
      cuuint32_t pbox[4] = {64, (cuuint32_t)(8 * num_shards), (cuuint32_t)kChunks, 1};
      cuuint32_t pes[4] = {1, (cuuint32_t)num_shards, 1, 1};
      if (encode(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(kv->data), pdims,
                 pstrides, pbox, pes, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MLA_ERR_CUDA;
    } else {
      cuuint64_t dims[5] = {64, 8, (cuuint64_t)kChunks, (cuuint64_t)(kPage / 8 / nv),
                            (cuuint64_t)kv->num_pages * kPage};
      cuuint64_t strides[4] = {(cuuint64_t)kDqk * nv, 64, (cuuint64_t)kDqk * 8 * nv,
                               (cuuint64_t)kDqk};
      cuuint32_t box[5] = {64, 8, (cuuint32_t)kChunks, (cuuint32_t)(kPage / 8 / nv), 1};
      cuuint32_t es[5] = {1, 1, 1, 1, 1};
      if (encode(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(kv->data), dims,
                 strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                 CU_TENSOR_MAP_L2_PROMOTION_NONE,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MLA_ERR_CUDA;
    }
  } else {
    cuuint64_t dims[5] = {64, 8, (cuuint64_t)kChunks, (cuuint64_t)(kPage / 8 / nv),
                          (cuuint64_t)kv->num_pages * kPage};
    cuuint64_t strides[4] = {(cuuint64_t)kDqk * 2 * nv, 128, (cuuint64_t)kDqk * 2 * 8 * nv,
                             (cuuint64_t)kDqk * 2};
    cuuint32_t box[5] = {64, 8, (cuuint32_t)kCgChunks, (cuuint32_t)(kPage / 8 / nv), 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    if (pd.pad) {
      // N does not divide 64: view (64 dims, row in page, chunk, page) with
      // strides (-, 1152, 128, 73728); a box of 8 N rows traversed with
      // stride N and three chunks lands one 8-slot group of a chunk group
      // (3072 bytes), and rows past the page's end fill zeros
      cuuint64_t pdims[4] = {64, (cuuint64_t)kPage, (cuuint64_t)kChunks,
                             (cuuint64_t)kv->num_pages};
      cuuint64_t pstrides[3] = {(cuuint64_t)kDqk * 2, 128, (cuuint64_t)kDqk * 2 * kPage};
      cuuint32_t pbox[4] = {64, (cuuint32_t)(8 * num_shards), (cuuint32_t)kCgChunks, 1};
      cuuint32_t pes[4] = {1, (cuuint32_t)num_shards, 1, 1};
      if (encode(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(kv->data),
                 pdims, pstrides, pbox, pes, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return MLA_ERR_CUDA;
    } else if (encode(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(kv->data),
                      dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
      return MLA_ERR_CUDA;
    }
    // the same view with all nine chunks in one box, for the L2 prefetch
    box[2] = (cuuint32_t)kChunks;
    if (encode(&tm_kv_pf, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(kv->data), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_CUDA;
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PartialParams p;
  p.pd = pd;
  p.out_partial = out_partial;
  p.lse_partial = lse_partial;
  p.hdr = reinterpret_cast<WsHeader*>(ws + wl.hdr);
  p.prefix = reinterpret_cast<int*>(ws + wl.prefix);
  p.ws_o = reinterpret_cast<float*>(ws + wl.ws_o);
  p.ws_lse = reinterpret_cast<float*>(ws + wl.ws_lse);
  p.kv_scale = kv->scale;
  p.q_one_box = q_one_box;
  p.kv_fp8 = nullptr;
  p.q = static_cast<const uint16_t*>(q);
  p.timeout_ns = host::wait_budget_ns(kTimeoutNs);
  p.withhold_query = host::g_withhold_query.load();

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_plan(pd, p.hdr, p.prefix, grid, kMinTilesPerCta, fp8 ? kUnitCostFp8 : kUnitCost,
                  st) != cudaSuccess)
    return MLA_ERR_CUDA;
  void* ev0 = host::g_ev_before.load();
  void* ev1 = host::g_ev_after.load();
  if (ev0 != nullptr && cudaEventRecord(static_cast<cudaEvent_t>(ev0), st) != cudaSuccess)
    return MLA_ERR_CUDA;
  const cudaError_t le = fp8 ? launch_partial_fp8(tm_q8, tm_kv, p, grid, st)
                             : launch_partial_bf16(tm_q, tm_kv, tm_kv_pf, p, grid, st);
  if (ev1 != nullptr && cudaEventRecord(static_cast<cudaEvent_t>(ev1), st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (le != cudaSuccess) return MLA_ERR_CUDA;
  L->pd = pd;
  L->hdr = p.hdr;
  L->prefix = p.prefix;
  L->ws_o = p.ws_o;
  L->ws_lse = p.ws_lse;
  L->num_units = U;
  return MLA_OK;
}

// Workspace of a whole decode step: the partial-attention workspace, the
// shard partials [N, B, R, 512] and their LSEs [N, B, R], then the combined
// output [B, R, 512] in bf16 that the tensor-core W_UV projection reads.
struct StepLayout {
  size_t partial_ws, part, part_lse, obf, total;
};

StepLayout step_layout(const mla_shape* shape, int num_shards) {
  auto up = [](size_t v) { return (v + 255) & ~static_cast<size_t>(255); };
  StepLayout s;
  s.partial_ws = up(mla_workspace_size(shape, num_shards, MLA_ALL_SHARDS));
  const size_t rows1 = (size_t)shape->batch * shape->q_len * shape->num_heads;
  const size_t rows = (size_t)num_shards * rows1;
  s.part = s.partial_ws;
  s.part_lse = s.part + up(rows * kDv * sizeof(float));
  s.obf = s.part_lse + up(rows * sizeof(float));
  s.total = s.obf + up(rows1 * kDv * sizeof(uint16_t));
  return s;
}

// Rows per head from which the fused W_UV projection runs as a tensor-core
// GEMM per head (after a combine that writes O) instead of on the CUDA cores
// inside the combine.
constexpr int kWuvGemmMinRows = 64;

}  // namespace

extern "C" {

mla_status mla_decode_partial(const void* q, const mla_kv_pages* kv, const int32_t* block_table,
                              int max_pages_per_req, const int32_t* seq_lens,
                              const mla_shape* shape, int shard_id, int num_shards,
                              mla_layout layout, float* out_partial, float* lse_partial,
                              void* workspace, size_t workspace_bytes, void* stream) {
  Launched L;
  const mla_status st = partial_launch(q, kv, block_table, max_pages_per_req, seq_lens, shape,
                                       shard_id, num_shards, layout, out_partial, lse_partial,
                                       workspace, workspace_bytes, stream, &L);
  if (st != MLA_OK) return st;
  if (launch_merge(L.pd, L.hdr, L.prefix, L.ws_o, L.ws_lse, out_partial, lse_partial,
                   L.num_units, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status mla_decode_partial_dcp(const void* q_gathered, int batch_total, int batch_first,
                                  const mla_kv_pages* kv, const int32_t* block_table,
                                  int max_pages_per_req, const int32_t* seq_lens,
                                  const mla_shape* shape, int rank, int num_ranks,
                                  mla_layout layout, float* out_send, float* lse_send,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  if (!shape_ok(shape) || num_ranks < 1 || num_ranks > kMaxShards || rank < 0 ||
      rank >= num_ranks)
    return MLA_ERR_INVALID;
  if (batch_first < 0 || batch_total < shape->batch ||
      batch_first > batch_total - shape->batch)
    return MLA_ERR_INVALID;
  if (shape->num_heads % num_ranks != 0) return MLA_ERR_INVALID;
  // a rank holds its own slice of the cache
  if (layout != MLA_LAYOUT_INTERLEAVED_LOCAL && layout != MLA_LAYOUT_CONTIGUOUS_LOCAL)
    return MLA_ERR_INVALID;
  const int hl = shape->num_heads / num_ranks;
  // runs of one rank's heads are whole 8-row groups, and a 64-row query
  // group is a whole number of runs (or lies inside one)
  if (hl % 8 != 0 || (kRows % hl != 0 && hl % kRows != 0)) return MLA_ERR_UNSUPPORTED;
  Launched L;
  const mla_status st = partial_launch(q_gathered, kv, block_table, max_pages_per_req, seq_lens,
                                       shape, rank, num_ranks, layout, out_send, lse_send,
                                       workspace, workspace_bytes, stream, &L,
                                       RankIo{hl, num_ranks, batch_total, batch_first});
  if (st != MLA_OK) return st;
  if (launch_merge(L.pd, L.hdr, L.prefix, L.ws_o, L.ws_lse, out_send, lse_send, L.num_units,
                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

size_t mla_decode_step_workspace_size(const mla_shape* shape, int num_shards) {
  if (mla_workspace_size(shape, num_shards, MLA_ALL_SHARDS) == 0) return 0;
  return step_layout(shape, num_shards).total;
}

mla_status mla_decode_step(const void* q, const mla_kv_pages* kv, const int32_t* block_table,
                           int max_pages_per_req, const int32_t* seq_lens, const mla_shape* shape,
                           int num_shards, mla_layout layout, const void* w_uv, void* out,
                           float* lse_out, void* workspace, size_t workspace_bytes,
                           void* stream) {
  if (out == nullptr || !aligned16(out) || (w_uv != nullptr && !aligned16(w_uv)) ||
      (lse_out != nullptr && !aligned4(lse_out)))
    return MLA_ERR_INVALID;
  if (!shape_ok(shape) || num_shards < 1 || num_shards > kMaxShards) return MLA_ERR_INVALID;
  if (layout != MLA_LAYOUT_INTERLEAVED && layout != MLA_LAYOUT_CONTIGUOUS) return MLA_ERR_INVALID;
  if (workspace == nullptr || !aligned16(workspace)) return MLA_ERR_WORKSPACE;
  const size_t need_partial = mla_workspace_size(shape, num_shards, MLA_ALL_SHARDS);
  if (need_partial == 0) return MLA_ERR_INVALID;
  const StepLayout sl = step_layout(shape, num_shards);
  if (workspace_bytes < sl.total) return MLA_ERR_WORKSPACE;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  float* part = reinterpret_cast<float*>(ws + sl.part);
  float* part_lse = reinterpret_cast<float*>(ws + sl.part_lse);
  Launched L;
  const mla_status st = partial_launch(q, kv, block_table, max_pages_per_req, seq_lens, shape,
                                       MLA_ALL_SHARDS, num_shards, layout, part, part_lse,
                                       workspace, sl.partial_ws, stream, &L);
  if (st != MLA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int rows_per_head = shape->batch * shape->q_len;
  if (w_uv != nullptr && rows_per_head >= kWuvGemmMinRows) {
    // many rows per head: the combine writes O (bf16) into the workspace and
    // one tcgen05 GEMM per head projects it
    uint16_t* obf = reinterpret_cast<uint16_t*>(ws + sl.obf);
    if (launch_step_combine(L.pd, L.hdr, L.prefix, L.ws_o, L.ws_lse, part, part_lse, nullptr,
                            obf, lse_out, cs) != cudaSuccess ||
        launch_wuv_gemm(obf, static_cast<const uint16_t*>(w_uv), static_cast<uint16_t*>(out),
                        rows_per_head, shape->num_heads, &L.hdr->err,
                        host::wait_budget_ns(kTimeoutNs), cs) != cudaSuccess)
      return MLA_ERR_CUDA;
    return MLA_OK;
  }
  if (launch_step_combine(L.pd, L.hdr, L.prefix, L.ws_o, L.ws_lse, part, part_lse,
                          static_cast<const uint16_t*>(w_uv), static_cast<uint16_t*>(out),
                          lse_out, cs) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status mla_shard_combine(const float* partials, const float* lses, int num_shards,
                             const mla_shape* shape, const void* w_uv, void* out, float* lse_out,
                             void* stream) {
  if (!partials || !lses || !out || !shape_ok(shape)) return MLA_ERR_INVALID;
  if (num_shards < 1 || num_shards > kMaxShards) return MLA_ERR_INVALID;
  if (!aligned16(partials) || !aligned16(out) || (w_uv && !aligned16(w_uv)) ||
      !aligned4(lses) || (lse_out && !aligned4(lse_out)))
    return MLA_ERR_INVALID;
  const int rows = shape->batch * shape->q_len * shape->num_heads;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (w_uv == nullptr)
    e = launch_combine(partials, lses, num_shards, rows, static_cast<uint16_t*>(out), lse_out, st);
  else
    e = launch_combine_wuv(partials, lses, num_shards, shape->batch * shape->q_len,
                           shape->num_heads, static_cast<const uint16_t*>(w_uv),
                           static_cast<uint16_t*>(out), lse_out, st);
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

mla_status mla_set_profile_events(void* before_partial, void* after_partial) {
  if ((before_partial == nullptr) != (after_partial == nullptr)) return MLA_ERR_INVALID;
  host::g_ev_before.store(before_partial);
  host::g_ev_after.store(after_partial);
  return MLA_OK;
}

mla_status mla_set_wait_budget_ns(unsigned long long ns) {
  host::g_wait_budget_ns.store(ns);
  return MLA_OK;
}

mla_status mla_set_withhold_query(int on) {
  host::g_withhold_query.store(on != 0 ? 1 : 0);
  return MLA_OK;
}

mla_status mla_get_device_error(void* workspace, void* stream) {
  if (workspace == nullptr) return MLA_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned err = 0;
  if (cudaMemcpyAsync(&err, workspace, sizeof(err), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  if (err != 0) {
    // cleared in stream order, behind everything already queued on `stream`
    if (cudaMemsetAsync(workspace, 0, sizeof(unsigned), st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  if (err & kErrTimeout) return MLA_ERR_TIMEOUT;
  if (err & kErrBadPage) return MLA_ERR_DEVICE_BOUNDS;
  if (err & kErrQRange) return MLA_ERR_RANGE;
  if (err & kErrQLens) return MLA_ERR_INVALID;
  return MLA_OK;
}

}  // extern "C"
