// kernels.cuh -- argument blocks and launchers shared between the C-ABI layer
// (api.cu) and the kernel translation units.
#pragma once
#include <cuda.h>

#include <atomic>

#include "common.cuh"

namespace kvq {

// Partitions per block of the fused merge's first level (kvq_decode_merged).
constexpr int kMergeBlock = 8;

// Split-T decode over the 4-bit rotated cache (decode_q4.cu).
struct DecodeArgs {
  CUtensorMap tm_k;  // 4-bit: K codes plane as [rows][128 B], 16-row boxes, 128-byte swizzle;
                     // fp8: latent codes [rows][512 B], 128 x 16 boxes, 128-byte swizzle
  CUtensorMap tm_v;  // 4-bit: V codes plane, same shape; fp8: rope codes [rows][64 B], 64-byte swizzle
  kvq_cache c;
  const float* q;  // [B, Hq, D] (4-bit: rotated; fp8: [B, Hq, 576])
  int Hq;
  int group;  // Hq / Hk
  const int32_t* seq_lens;
  const int32_t* block_tables;
  int max_pages;
  int max_seq_len;
  const int32_t* sel;  // NULL: dense
  int n_sel;
  float qscale;  // sm_scale * log2(e)
  const void* q_raw;  // 4-bit format only: unrotated query [B, Hq, 256] of q_dtype, rotated in
                      // the kernel (then q is unused); NULL: q is already rotated
  int q_dtype;
  int q_rotate;       // q_raw only: 1 rotate it (Hadamard format), 0 use it as given (Q4_0)
  float* ws_m;
  float* ws_z;
  float* ws_acc;
  int P;  // partitions per (seq, head) in the workspace
  int32_t* status;
  // 4-bit decode only.  Block-table row of sequence b: block_tables + b * bt_stride
  // (bt_stride 0: one table shared by every row of a decode window).  nrows > 0:
  // a decode window of nrows rows (seq_lens holds each row's length), cut into
  // slices of rows_per_cta rows (set by the launch) whose (row, head) pairs one
  // CTA scores together; nrows = 0: one sequence per CTA.
  int bt_stride;
  int nrows;
  int rows_per_cta;
  int tq;  // 4-bit decode: 1 for TQ4 rows (codebook levels, one scale per row)
  int part;  // keys per partition (512; the fp8 streaming prefill: a whole row)
  // fp8 prefill chunk: row b is the query at position prefill_q0 + b and attends
  // keys 0 .. prefill_q0 + b (seq_lens unused); 0: decode
  int prefill;
  int prefill_q0;
  // 4-bit decode with the fused merge: the merged outputs [B][Hq][256]; the
  // completion counters (zero between launches): [B][Hk] per (sequence, KV
  // head), then [B][Hk][merge_nblk] per block of 8 partitions; the block
  // partials m, z [B][Hq][merge_nblk] and acc [B][Hq][merge_nblk][256]
  float* fused_out;
  int32_t* merge_ctr;
  int merge_B;
  int merge_nblk;
  float* merge_m;
  float* merge_z;
  float* merge_acc;
  // 4-bit dense decode (kvq_decode_step): each sequence's new K and V rows
  // [B][Hk][256] of new_dtype, stored at position seq_lens[b] - 1 by the CTA whose
  // partition holds it before that CTA reads its tiles; NULL: nothing to store
  const void* new_k;
  const void* new_v;
  int new_dtype;
};

// Log-sum-exp merge of the partials (merge.cu).
struct MergeArgs {
  const float* ws_m;
  const float* ws_z;
  const float* ws_acc;
  int P;
  int Hq;
  int Dv;
  const int32_t* seq_lens;
  int max_seq_len;
  int n_sel;
  int rotate_back;
  float* out;
  int part;  // keys per partition (as in the decode that wrote the partials)
  int prefill;     // 1: row b has prefill_q0 + b + 1 keys (seq_lens unused)
  int prefill_q0;
};

// Causal prefill over decoded 4-bit slots (prefill_tc.cu).
struct PrefillArgs {
  CUtensorMap tm_k;  // 4-bit: K codes plane as [rows][128 B], 16-row boxes, 128-byte swizzle;
                     // fp8: latent codes [rows][512 B], 128 x 16 boxes, 128-byte swizzle
  CUtensorMap tm_v;  // 4-bit: V codes plane, same shape; fp8: rope codes [rows][64 B], 64-byte swizzle
  kvq_cache c;
  const void* q;
  int dtype;
  int n_q;
  int Hq;
  int group;
  int q_start;
  const int32_t* block_table;
  int max_pages;
  float qscale;
  float* out;
  int32_t* status;
  int rotate;  // 1: Hadamard format (rotate q, rotate the output back); 0: Q4_0
};

// The host-side checks of kvq_decode_attn + kvq_merge on a workspace of ws_bytes
// bytes (api.cu); enqueues nothing.
int32_t check_decode_and_merge(const kvq_cache* cache, const float* q, int32_t num_seqs, int32_t num_q_heads,
                               const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                               int32_t max_seq_len, const int32_t* d_sel, int32_t n_sel, int32_t rotate_back,
                               const float* out, size_t ws_bytes);

// Remember a failed CUDA call for kvq_last_cuda_error(); returns KVQ_ERR_CUDA.
int32_t record_cuda_failure(cudaError_t e);

// ---------------------------------------------------------------- per-launch invariants (host.cu)
// Unique ID of the calling thread's current CUDA context (0 if there is none or
// it cannot be read).  A context re-created by cudaDeviceReset, or another
// context made current, has another ID.
unsigned long long current_context_id();
// Streaming multiprocessors of the current device (queried once per device).
int device_sm_count();

// Raise Kern's dynamic shared-memory limit to `bytes`, once per CUDA context
// (the attribute lives as long as the context; a context of another ID, or one
// whose ID cannot be read, sets it again).
template <auto Kern>
cudaError_t set_max_smem_once(int bytes) {
  static std::atomic<unsigned long long> done_ctx{0};
  const unsigned long long ctx = current_context_id();
  if (ctx != 0 && done_ctx.load(std::memory_order_acquire) == ctx) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && ctx != 0) done_ctx.store(ctx, std::memory_order_release);
  return e;
}

cudaError_t launch_store(const kvq_cache& c, const void* k, const void* v, int dtype, int64_t n_tok,
                         const int32_t* slots, int32_t* status, cudaStream_t s);
cudaError_t launch_rotate(const void* x, int dtype, float* y, int64_t rows, int head_dim, cudaStream_t s);
// kvq_store (the few-row 4-bit form) and kvq_rotate_query in one launch.
bool store_rotate_fits(const kvq_cache& c, int64_t n_tok);
cudaError_t launch_store_rotate(const kvq_cache& c, const void* k, const void* v, int dtype, int64_t n_tok,
                                const int32_t* slots, int32_t* status, const void* q, int q_dtype, float* q_out,
                                int64_t q_rows, int q_head_dim, cudaStream_t s);
cudaError_t launch_decode_q4(const DecodeArgs& a, int B, cudaStream_t s);
// Whether a dense 4-bit decode grid of `ctas` CTAs runs in one wave (two CTAs per SM).
bool decode_q4_one_wave(int64_t ctas);
// TQ4 rows (tq4.cu): store, and the signed row rotation (inverse = 1: outputs back).
cudaError_t launch_store_tq4(const kvq_cache& c, const void* k, const void* v, int dtype, int64_t n_tok,
                             const int32_t* slots, int32_t* status, cudaStream_t s);
cudaError_t launch_tq4_rotate(const kvq_cache& c, const void* x, int dtype, float* y, int64_t rows, int inverse,
                              cudaStream_t s);
// fp8 latent rows on the tensor cores (decode_fp8.cu); tm_k / tm_v map the latent
// and rope code planes.
cudaError_t launch_decode_fp8(const DecodeArgs& a, int B, cudaStream_t s);
// bf16 rows on the tensor cores (decode_bf16.cu); tm_k / tm_v map the K and V
// planes as [rows][512 B] in 128-byte column boxes.
cudaError_t launch_decode_bf16(const DecodeArgs& a, int B, cudaStream_t s);
cudaError_t launch_merge(const MergeArgs& a, int B, cudaStream_t s);
// A barrier wait that nothing completes, bounded like every copy wait (api.cu).
cudaError_t launch_wait_timeout_probe(int32_t* status, cudaStream_t s);
cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s);

}  // namespace kvq
