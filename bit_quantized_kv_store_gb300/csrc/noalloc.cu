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
// loading this library holds until the process exits.  Host code cannot use the
// array's name as a device address: its address is looked up with
// cudaGetSymbolAddress, with the device current, and cached per device together
// with the unique ID of the CUDA context it was looked up in.  A call made in
// another context (a non-primary context the caller made current, or the
// primary context re-created after cudaDeviceReset) looks the address up again.
// This translation unit is its own module, which CUDA loads lazily: the first
// lookup in a context loads it and commits the 16 MiB there, so that first call
// must come outside any region where the caller cannot allocate, and before any
// stream capture.  Every call shares the array and the array keeps the last
// call's contents: the status word is cleared on the stream at the start of each
// call, and calls whose work overlaps on the GPU (different streams without
// ordering) race on it.
#include <cudaTypedefs.h>

#include <mutex>

#include "kernels.cuh"

namespace kvq {

constexpr size_t kKvqStaticScratchBytes = size_t(16) << 20;

static __device__ __align__(256) uint8_t g_static_scratch[kKvqStaticScratchBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  unsigned long long ctx_id;  // unique ID of the context the address belongs to (0: none yet)
  void* ptr;
};
static ScratchAddr g_scratch[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of the scratch array in the current device's current context.
static cudaError_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long id = current_context_id();
  if (id != 0 && g_scratch[dev].ctx_id == id) {
    *out = g_scratch[dev].ptr;
    return cudaSuccess;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_scratch);  // binds the primary context if none was current
  if (e != cudaSuccess) return e;
  if (id == 0) id = current_context_id();
  g_scratch[dev] = ScratchAddr{id, id != 0 ? p : nullptr};
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
  if (cache == nullptr) return KVQ_ERR_INVALID_ARG;
  const int32_t ns = d_sel ? n_sel : 0;
  if (kvq_decode_workspace_size(cache, num_seqs, num_q_heads, max_seq_len, ns) == 0) return KVQ_ERR_INVALID_ARG;
  // every check of the two calls below, before anything is enqueued
  int32_t st = check_decode_and_merge(cache, q, num_seqs, num_q_heads, d_seq_lens, d_block_tables, max_pages_per_seq,
                                      max_seq_len, d_sel, ns, rotate_back, out, kKvqStaticScratchBytes);
  if (st != KVQ_OK) return st;
  if (num_seqs == 0) return KVQ_OK;
  void* ws = nullptr;
  cudaError_t e = static_scratch(&ws);
  if (e != cudaSuccess) return record_cuda_failure(e);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(ws, 0, sizeof(int32_t), s);  // the status word must start at zero
  if (e != cudaSuccess) return record_cuda_failure(e);
  st = kvq_decode_attn(cache, q, num_seqs, num_q_heads, d_seq_lens, d_block_tables, max_pages_per_seq, max_seq_len,
                       d_sel, ns, sm_scale, ws, kKvqStaticScratchBytes, stream);
  if (st != KVQ_OK) return st;
  st = kvq_merge(cache, ws, kKvqStaticScratchBytes, num_seqs, num_q_heads, d_seq_lens, max_seq_len, ns, rotate_back,
                 out, stream);
  if (st != KVQ_OK) return st;
  if (d_status_out) {
    e = cudaMemcpyAsync(d_status_out, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return record_cuda_failure(e);
  }
  return KVQ_OK;
}

}  // extern "C"
