// host.cu -- host-side caches of per-launch invariants: the current context's
// ID (for keying anything that a context owns) and the SM count per device.
#include <cudaTypedefs.h>

#include "kernels.cuh"

namespace kvq {

// cuCtxGetCurrent / cuCtxGetId through the runtime's driver entry points (no
// link-time dependency on libcuda); looked up once.
struct CtxQueries {
  PFN_cuCtxGetCurrent_v4000 current = nullptr;
  PFN_cuCtxGetId_v12000 id = nullptr;
};
static const CtxQueries& ctx_queries() {
  static const CtxQueries q = [] {
    CtxQueries r;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult st;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &st) == cudaSuccess &&
        st == cudaDriverEntryPointSuccess)
      r.current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &st) == cudaSuccess &&
        st == cudaDriverEntryPointSuccess)
      r.id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    return r;
  }();
  return q;
}

unsigned long long current_context_id() {
  const CtxQueries& q = ctx_queries();
  if (!q.current || !q.id) return 0;
  CUcontext ctx = nullptr;
  if (q.current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (q.id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int device_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> counts[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) {
    const int n = counts[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < kMaxDevices) counts[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace kvq
