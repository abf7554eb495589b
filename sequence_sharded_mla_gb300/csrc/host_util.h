// Host-side helpers shared by the C ABI translation units: tensor-map
// encoding through the driver entry point, the SM count, pointer alignment
// and the profiling events of mla_set_profile_events.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

namespace mla {
namespace host {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// int32 index arrays (block table, lengths) are read one element at a time
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

inline int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// cudaEvent_t handles recorded around every partial-attention kernel launch
// while set (mla_set_profile_events).
inline std::atomic<void*> g_ev_before{nullptr}, g_ev_after{nullptr};

// Time limit of every device-side wait, in ns, for launches made from now
// on (mla_set_wait_budget_ns); 0 selects each kernel's default.
inline std::atomic<unsigned long long> g_wait_budget_ns{0};
inline unsigned long long wait_budget_ns(unsigned long long dflt) {
  const unsigned long long v = g_wait_budget_ns.load();
  return v != 0 ? v : dflt;
}

// Testing aid (mla_set_withhold_query): while non-zero, partial-attention
// launches never load the query rows of each CTA's first piece, so the waits
// for them can only run out.
inline std::atomic<int> g_withhold_query{0};

// Unique id of the CUDA context current on the calling thread (the device's
// primary context for runtime users), made current first if none is.  Ids
// are never reused within a process, so per-context state keyed on them
// stays correct across cudaDeviceReset and for contexts created through the
// driver API.  Returns 0 if it cannot be determined.
inline unsigned long long current_context_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static const GetCurrentFn get_current = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    return (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
               ? reinterpret_cast<GetCurrentFn>(f)
               : nullptr;
  }();
  static const GetIdFn get_id = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    return (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
               ? reinterpret_cast<GetIdFn>(f)
               : nullptr;
  }();
  if (get_current == nullptr || get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return 0;
  if (ctx == nullptr) {
    // no context yet: cudaSetDevice initialises the device's primary context
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return 0;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// A small table of values keyed by (context id, key), guarded by a mutex,
// for host-side state that belongs to one context: attributes set on a
// kernel, device addresses of module symbols.
template <class T, int kSlots = 64>
class PerContext {
 public:
  // Value for (context, key), computed by make() on first use.  make()
  // returns false on failure; nothing is stored then.
  template <class Make>
  bool get(const void* key, T& out, Make make) {
    const unsigned long long ctx = current_context_id();
    if (ctx == 0) return false;
    std::lock_guard<std::mutex> lock(mutex_);
    for (int i = 0; i < used_; ++i)
      if (slots_[i].ctx == ctx && slots_[i].key == key) {
        out = slots_[i].value;
        return true;
      }
    T v{};
    if (!make(v)) return false;
    const int i = used_ < kSlots ? used_++ : (next_evict_++ % kSlots);
    slots_[i] = Slot{ctx, key, v};
    out = v;
    return true;
  }

 private:
  struct Slot {
    unsigned long long ctx;
    const void* key;
    T value;
  };
  std::mutex mutex_;
  Slot slots_[kSlots] = {};
  int used_ = 0;
  int next_evict_ = 0;
};

// Raises a kernel's dynamic shared-memory limit once per context (the
// attribute belongs to the context's copy of the module).
inline cudaError_t ensure_dynamic_smem(const void* kernel, int bytes) {
  static PerContext<int> done;
  int ok = 0;
  cudaError_t err = cudaSuccess;
  if (!done.get(kernel, ok, [&](int& v) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        v = 1;
        return err == cudaSuccess;
      }))
    return err != cudaSuccess ? err : cudaErrorInitializationError;
  return cudaSuccess;
}

}  // namespace host
}  // namespace mla
