// mla_decode_partial_noalloc: the per-shard partial attention call for
// callers that must not allocate device memory.
//
// mla_decode_partial needs a caller-provided workspace (the work list and the
// partial results of work units that are split across CTAs).  Some callers
// cannot obtain one: code that runs while every byte of the GPU is already
// owned by a serving engine's memory pool, code inside allocator callbacks or
// out-of-memory handlers, latency-critical loops where an allocation (and the
// synchronisation it may imply) is not allowed, and hosts in other languages
// that have no handle on the framework's allocator.  For them this file keeps
// one fixed scratch buffer per GPU in a file-scope __device__ array and runs
// the ordinary partial-attention path on it.  Nothing here allocates.
#include <cuda_runtime.h>

#include "common.cuh"
#include "host_util.h"
#include "mla_dcp.h"

namespace {

// Largest workspace this entry point can serve: the 256-byte header, the tile
// prefix of up to kMaxUnits work units, and two split-piece slots
// (64 rows x 512 fp32 output + 64 fp32 LSE) for each of up to kMaxCtas
// persistent CTAs.  The grid of the partial kernel is one CTA per SM, so the
// slots cover GPUs with up to 160 SMs.
constexpr size_t kMaxUnits = 8192;
constexpr size_t kMaxCtas = 160;
constexpr size_t kScratchBytes =
    256 + 256 * ((sizeof(int) * (kMaxUnits + 1) + 255) / 256) +
    kMaxCtas * 2 * mla::kRows * mla::kDv * sizeof(float) + kMaxCtas * 2 * mla::kRows * sizeof(float);

// The scratch itself: every GPU that loads this library holds one copy until
// the process exits (about 40 MiB).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Device address of the scratch in the current context.  The host-side
// symbol is only a stand-in; kernels must be given the address that
// cudaGetSymbolAddress returns, looked up once per CUDA context (a new
// context after cudaDeviceReset, or a driver-API context, holds its own copy
// of the module and so its own scratch).
void* scratch_for_current_context() {
  static mla::host::PerContext<void*> table;
  void* ptr = nullptr;
  if (!table.get(reinterpret_cast<const void*>(&g_noalloc_scratch), ptr, [](void*& v) {
        v = nullptr;
        return cudaGetSymbolAddress(&v, g_noalloc_scratch) == cudaSuccess && v != nullptr;
      }))
    return nullptr;
  return ptr;
}

}  // namespace

extern "C" mla_status mla_decode_partial_noalloc(const void* q, const mla_kv_pages* kv,
                                                 const int32_t* block_table,
                                                 int max_pages_per_req, const int32_t* seq_lens,
                                                 const mla_shape* shape, int shard_id,
                                                 int num_shards, mla_layout layout,
                                                 float* out_partial, float* lse_partial,
                                                 void* stream) {
  if (shape == nullptr || num_shards < 1 || num_shards > mla::kMaxShards) return MLA_ERR_INVALID;
  if (shape->batch < 1 || shape->q_len < 1 || shape->num_heads < 1) return MLA_ERR_INVALID;
  // The stated limits, checked with host arithmetic before any CUDA call.
  const long long n_out = shard_id == MLA_ALL_SHARDS ? num_shards : 1;
  const long long groups = ((long long)shape->q_len * shape->num_heads + mla::kRows - 1) / mla::kRows;
  if ((long long)shape->batch * n_out * groups > (long long)kMaxUnits) return MLA_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (sms > (int)kMaxCtas) return MLA_ERR_UNSUPPORTED;
  const size_t need = mla_workspace_size(shape, num_shards, shard_id);
  if (need == 0) return MLA_ERR_INVALID;
  if (need > kScratchBytes) return MLA_ERR_UNSUPPORTED;  // cannot happen within the limits
  void* scratch = scratch_for_current_context();
  if (scratch == nullptr) return MLA_ERR_CUDA;
  // Everything the kernels read from the scratch is written earlier in the
  // same call (the planning kernel resets the error word and rebuilds the
  // work list), so the previous call's contents need no clearing here.
  return mla_decode_partial(q, kv, block_table, max_pages_per_req, seq_lens, shape, shard_id,
                            num_shards, layout, out_partial, lse_partial, scratch, kScratchBytes,
                            stream);
}

// The error word of the scratch (its first four bytes, as in every
// workspace), read and cleared on `stream` exactly as mla_get_device_error
// does for a caller's workspace.
extern "C" mla_status mla_get_device_error_noalloc(void* stream) {
  void* scratch = scratch_for_current_context();
  if (scratch == nullptr) return MLA_ERR_CUDA;
  return mla_get_device_error(scratch, stream);
}
