// noalloc.cu -- a decode entry point that needs no caller-provided workspace.
//
// kvq_decode_attn + kvq_merge need a workspace for the split-T partials, which
// the caller allocates.  Some callers cannot allocate device memory at the
// point where they decode: code running inside a memory pool that forbids
// new allocations, plug-ins of hosts that own every device allocation, or
// real-time paths where cudaMalloc's implicit synchronisation and latency are
// not acceptable.  kvq_decode_noalloc serves them: it runs the same two kernels
// with the partials in a fixed, file-scope device array instead.
//
// The array is kKvqStaticScratchBytes (16 MiB) of device memory that every GPU
// loading this library holds until the process exits.  Its device address is
// looked up once per device (cudaGetSymbolAddress with that device current) on
// the first call made on that device; make that first call before any stream
// capture begins.  Every call shares the array and the array keeps the last
// call's contents: the status word is cleared on the stream at the start of each
// call, and calls whose work overlaps on the GPU (different streams or devices
// sharing a context without ordering) race on it.
#include <atomic>
#include <mutex>

#include "kernels.cuh"

namespace kvq {

constexpr size_t kKvqStaticScratchBytes = size_t(16) << 20;

static __device__ __align__(256) uint8_t g_static_scratch[kKvqStaticScratchBytes];

constexpr int kMaxDevices = 64;
static std::atomic<void*> g_scratch_ptr[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once).
static cudaError_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_static_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace kvq

using namespace kvq;

extern "C" {

size_t kvq_noalloc_scratch_bytes(void) { return kKvqStaticScratchBytes; }

int32_t kvq_decode_noalloc(const kvq_cache* cache, const float* q, int32_t num_seqs, int32_t num_q_heads,
                           const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                           int32_t max_seq_len, const int32_t* d_sel, int32_t n_sel, float sm_scale,
                           int32_t rotate_back, float* out, int32_t* d_status_out, void* stream) {
  const size_t need = kvq_decode_workspace_size(cache, num_seqs, num_q_heads, max_seq_len, d_sel ? n_sel : 0);
  if (cache == nullptr || need == 0) return KVQ_ERR_INVALID_ARG;
  if (need > kKvqStaticScratchBytes) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  if (num_seqs == 0) return KVQ_OK;
  if (!out) return KVQ_ERR_INVALID_ARG;
  void* ws = nullptr;
  cudaError_t e = static_scratch(&ws);
  if (e != cudaSuccess) return record_cuda_failure(e);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(ws, 0, sizeof(int32_t), s);  // the status word must start at zero
  if (e != cudaSuccess) return record_cuda_failure(e);
  int32_t st = kvq_decode_attn(cache, q, num_seqs, num_q_heads, d_seq_lens, d_block_tables, max_pages_per_seq,
                               max_seq_len, d_sel, d_sel ? n_sel : 0, sm_scale, ws, kKvqStaticScratchBytes, stream);
  if (st != KVQ_OK) return st;
  st = kvq_merge(cache, ws, kKvqStaticScratchBytes, num_seqs, num_q_heads, d_seq_lens, max_seq_len,
                 d_sel ? n_sel : 0, rotate_back, out, stream);
  if (st != KVQ_OK) return st;
  if (d_status_out) {
    e = cudaMemcpyAsync(d_status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return record_cuda_failure(e);
  }
  return KVQ_OK;
}

}  // extern "C"
