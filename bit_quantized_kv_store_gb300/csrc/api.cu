// api.cu -- the C ABI of libkvq (declared in include/kvq.h): host-side argument
// validation, workspace geometry and kernel launches.  Nothing here allocates.
#include <cudaTypedefs.h>

#include <cstdio>

#include <mutex>

#include "kernels.cuh"

namespace kvq {

static thread_local int32_t g_last_cuda_error = 0;

static int32_t cuda_fail(cudaError_t e) {
  g_last_cuda_error = static_cast<int32_t>(e);
  return KVQ_ERR_CUDA;
}

int32_t record_cuda_failure(cudaError_t e) { return cuda_fail(e); }

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The two 4-bit formats share planes, layout and kernels (Q4_0 without the rotation).
static bool is_q4(int32_t f) { return f == KVQ_FMT_Q4_HAD32 || f == KVQ_FMT_Q4_0; }

static size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Validate a cache description; returns KVQ_OK or a negative status.
static int32_t check_cache(const kvq_cache* c) {
  if (!c) return KVQ_ERR_INVALID_ARG;
  if (c->format < KVQ_FMT_Q4_HAD32 || c->format > KVQ_FMT_TQ4) return KVQ_ERR_INVALID_ARG;
  if (c->num_kv_heads < 1 || c->head_dim <= 0 || c->page_size <= 0 || c->num_pages < 0)
    return KVQ_ERR_INVALID_ARG;
  if (c->head_dim % 32 != 0) return KVQ_ERR_UNSUPPORTED;  // rows are built from 32-value groups
  if (c->page_size % 16 != 0) return KVQ_ERR_UNSUPPORTED;
  if (!c->k || !c->v || !aligned16(c->k) || !aligned16(c->v)) return KVQ_ERR_INVALID_ARG;
  if (is_q4(c->format)) {
    if (!c->k_scale || !c->v_scale || !aligned16(c->k_scale) || !aligned16(c->v_scale)) return KVQ_ERR_INVALID_ARG;
    const int ng = c->head_dim / 32;
    if (ng != 1 && ng != 2 && ng != 4 && ng != 8) return KVQ_ERR_UNSUPPORTED;
    if (c->rope_dim != 0) return KVQ_ERR_INVALID_ARG;
  } else if (c->format == KVQ_FMT_TQ4) {
    if (!c->k_scale || !c->v_scale || !aligned16(c->k_scale) || !aligned16(c->v_scale)) return KVQ_ERR_INVALID_ARG;
    if (!c->signs || (reinterpret_cast<uintptr_t>(c->signs) & 3u) != 0) return KVQ_ERR_INVALID_ARG;
    if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
    if (c->rope_dim != 0) return KVQ_ERR_INVALID_ARG;
  } else if (c->format == KVQ_FMT_BF16) {
    if (c->rope_dim != 0) return KVQ_ERR_INVALID_ARG;
  } else {
    if (c->num_kv_heads != 1 || c->rope_dim <= 0 || c->rope_dim % 16 != 0) return KVQ_ERR_INVALID_ARG;
    if (!c->k_scale || !c->v_scale) return KVQ_ERR_INVALID_ARG;
  }
  return KVQ_OK;
}

static int value_width(const kvq_cache* c) { return c->head_dim; }

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time
// dependency on libcuda); the pointer is looked up once.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// A plane of `rows` rows of `row_bytes` bytes as a 2-D byte tensor; boxes of
// box_bytes x box_rows with the given swizzle (box_bytes = the swizzle span).
// A tensor map holds nothing but the address and this geometry, so encoded maps
// are kept (the last kMapCache of them, under a lock) and a call on the same
// plane reuses one instead of encoding it again.
namespace {
struct MapKey {
  const void* base;
  uint64_t rows;
  uint32_t row_bytes, box_rows, box_bytes;
  int swizzle;
  bool operator==(const MapKey& o) const {
    return base == o.base && rows == o.rows && row_bytes == o.row_bytes && box_rows == o.box_rows &&
           box_bytes == o.box_bytes && swizzle == o.swizzle;
  }
};
constexpr int kMapCache = 64;
struct MapCache {
  std::mutex mu;
  MapKey key[kMapCache] = {};
  CUtensorMap map[kMapCache];
  bool used[kMapCache] = {};
  int next = 0;
};
MapCache& map_cache() {
  static MapCache c;
  return c;
}
}  // namespace

static bool encode_rows_map(CUtensorMap* m, const void* base, uint64_t rows, uint32_t row_bytes, uint32_t box_rows,
                            uint32_t box_bytes = 128, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  const MapKey key{base, rows, row_bytes, box_rows, box_bytes, static_cast<int>(swizzle)};
  MapCache& mc = map_cache();
  std::lock_guard<std::mutex> lock(mc.mu);
  for (int i = 0; i < kMapCache; ++i)
    if (mc.used[i] && mc.key[i] == key) {
      *m = mc.map[i];
      return true;
    }
  PFN_cuTensorMapEncodeTiled_v12000 fn = tensor_map_encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows > 0 ? rows : 1};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t es[2] = {1, 1};
  if (fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const int slot = mc.next;
  mc.next = (mc.next + 1) % kMapCache;
  mc.key[slot] = key;
  mc.map[slot] = *m;
  mc.used[slot] = true;
  return true;
}

struct WsLayout {
  size_t m_off, z_off, acc_off, ctr_off, bm_off, bz_off, bacc_off, total;
  int P;
  int part;  // keys per partition
  int nblk;  // the fused merge's blocks of kMergeBlock partitions
};

// Keys per split-T partition: 512 ("shared 512-key chunks") for every format
// and problem size, so that a sequence's partials do not depend on what else
// is in the batch (a batched sequence equals its solo decode bit for bit).
// A gather over selected fp8 latent rows takes runs of kFp8GatherPart entries
// instead: a selection of a few thousand rows would otherwise give a handful of
// CTAs per head block.
constexpr int kFp8GatherPart = 64;

static WsLayout ws_layout(const kvq_cache* c, int B, int Hq, int max_seq_len, int n_sel) {
  WsLayout w;
  const int64_t T = n_sel > 0 ? n_sel : max_seq_len;
  w.part = (n_sel > 0 && c->format == KVQ_FMT_FP8_ROW) ? kFp8GatherPart : kPart;
  w.P = static_cast<int>((T + w.part - 1) / w.part);
  if (w.P < 1) w.P = 1;
  const size_t n = static_cast<size_t>(B) * Hq * w.P;
  w.m_off = 256;
  w.z_off = w.m_off + round256(n * sizeof(float));
  w.acc_off = w.z_off + round256(n * sizeof(float));
  w.ctr_off = w.acc_off + round256(n * value_width(c) * sizeof(float));
  // the fused merge: completion counters per (sequence, KV head) and per block
  // of kMergeBlock partitions, then the block partials
  w.nblk = (w.P + kMergeBlock - 1) / kMergeBlock;
  const size_t nb = static_cast<size_t>(B) * Hq * w.nblk;
  w.bm_off = w.ctr_off + round256(static_cast<size_t>(B) * c->num_kv_heads * (1 + w.nblk) * sizeof(int32_t));
  w.bz_off = w.bm_off + round256(nb * sizeof(float));
  w.bacc_off = w.bz_off + round256(nb * sizeof(float));
  w.total = w.bacc_off + round256(nb * value_width(c) * sizeof(float));
  return w;
}

// Shared checks of the decode and merge arguments.
static int32_t check_decode_shape(const kvq_cache* c, int B, int Hq, const int32_t* seq_lens, int max_seq_len,
                                  bool gather, int n_sel) {
  if (B < 0 || Hq < 1 || max_seq_len < 0) return KVQ_ERR_INVALID_ARG;
  if (Hq % c->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (B > 0 && !seq_lens) return KVQ_ERR_INVALID_ARG;
  if (gather && (n_sel < 1 || n_sel > 4096)) return KVQ_ERR_INVALID_ARG;
  if (!gather && n_sel != 0) return KVQ_ERR_INVALID_ARG;
  const int group = Hq / c->num_kv_heads;
  if (c->format == KVQ_FMT_TQ4 && gather) return KVQ_ERR_UNSUPPORTED;
  if (is_q4(c->format) || c->format == KVQ_FMT_BF16 || c->format == KVQ_FMT_TQ4) {
    if (c->head_dim != 256 || group > 8) return KVQ_ERR_UNSUPPORTED;
  } else {
    if (c->head_dim != 512 || c->rope_dim != 64 || Hq % 16 != 0) return KVQ_ERR_UNSUPPORTED;
  }
  return KVQ_OK;
}

// The host-side checks of kvq_decode_attn followed by kvq_merge on one
// workspace of ws_bytes bytes, without enqueuing anything (used by the entry
// point whose workspace is the library's own scratch array, so that an invalid
// call leaves no work behind).
int32_t check_decode_and_merge(const kvq_cache* cache, const float* q, int32_t num_seqs, int32_t num_q_heads,
                               const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                               int32_t max_seq_len, const int32_t* d_sel, int32_t n_sel, int32_t rotate_back,
                               const float* out, size_t ws_bytes) {
  int32_t st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_sel < 0 || n_sel > 4096) return KVQ_ERR_INVALID_ARG;
  st = check_decode_shape(cache, num_seqs, num_q_heads, d_seq_lens, max_seq_len, d_sel != nullptr, n_sel);
  if (st != KVQ_OK) return st;
  if (rotate_back && cache->format != KVQ_FMT_Q4_HAD32 && cache->format != KVQ_FMT_TQ4) return KVQ_ERR_INVALID_ARG;
  if (num_seqs == 0) return KVQ_OK;
  if (!q || !aligned16(q) || !d_block_tables || max_pages_per_seq < 1 || !out) return KVQ_ERR_INVALID_ARG;
  if (!d_sel && static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages_per_seq) * cache->page_size)
    return KVQ_ERR_INVALID_ARG;
  if (ws_bytes < ws_layout(cache, num_seqs, num_q_heads, max_seq_len, d_sel ? n_sel : 0).total)
    return KVQ_ERR_WORKSPACE_TOO_SMALL;
  if (!d_sel && static_cast<uint64_t>(cache->num_pages) * cache->num_kv_heads * cache->page_size >= (1ull << 31))
    return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

}  // namespace kvq

using namespace kvq;

extern "C" {

int32_t kvq_version(void) { return 100; }

const char* kvq_status_string(int32_t s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape or format";
    case KVQ_ERR_CUDA: return "CUDA error";
    case KVQ_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    default: return "unknown status";
  }
}

int32_t kvq_last_cuda_error(void) { return g_last_cuda_error; }

size_t kvq_plane_bytes(const kvq_cache* c, int32_t plane) {
  if (!c || c->head_dim <= 0 || c->head_dim % 32 || c->num_kv_heads < 1 || c->page_size <= 0 || c->num_pages < 0)
    return 0;
  const size_t rows = static_cast<size_t>(c->num_pages) * c->num_kv_heads * c->page_size;
  switch (c->format) {
    case KVQ_FMT_Q4_HAD32:
    case KVQ_FMT_Q4_0:
      return (plane == 0 || plane == 2) ? rows * (c->head_dim / 2) : rows * (c->head_dim / 32) * 2;
    case KVQ_FMT_BF16:
      return (plane == 0 || plane == 2) ? rows * c->head_dim * 2 : 0;
    case KVQ_FMT_TQ4:
      return (plane == 0 || plane == 2) ? rows * (c->head_dim / 2) : rows * 2;
    case KVQ_FMT_FP8_ROW:
      if (plane == 0) return rows * c->head_dim;
      if (plane == 2) return rows * c->rope_dim;
      return rows * 4;
    default:
      return 0;
  }
}

int32_t kvq_store(const kvq_cache* cache, const void* k, const void* v, int32_t dtype, int64_t n_tok,
                  const int32_t* d_slot_mapping, int32_t* d_status, void* stream) {
  int32_t st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_tok < 0 || (dtype != KVQ_DT_F32 && dtype != KVQ_DT_BF16)) return KVQ_ERR_INVALID_ARG;
  if (n_tok == 0) return KVQ_OK;
  if (!k || !d_slot_mapping) return KVQ_ERR_INVALID_ARG;
  if (cache->format == KVQ_FMT_FP8_ROW) {
    if (v) return KVQ_ERR_INVALID_ARG;
  } else if (!v) {
    return KVQ_ERR_INVALID_ARG;
  }
  cudaError_t e = cache->format == KVQ_FMT_TQ4
                      ? launch_store_tq4(*cache, k, v, dtype, n_tok, d_slot_mapping, d_status,
                                         static_cast<cudaStream_t>(stream))
                      : launch_store(*cache, k, v, dtype, n_tok, d_slot_mapping, d_status,
                                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

int32_t kvq_tq4_rotate(const kvq_cache* cache, const void* x, int32_t dtype, float* y, int64_t rows,
                       int32_t inverse, void* stream) {
  int32_t st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (cache->format != KVQ_FMT_TQ4) return KVQ_ERR_UNSUPPORTED;
  if (rows < 0 || (dtype != KVQ_DT_F32 && dtype != KVQ_DT_BF16)) return KVQ_ERR_INVALID_ARG;
  if (rows == 0) return KVQ_OK;
  if (!x || !y) return KVQ_ERR_INVALID_ARG;
  if (x == static_cast<const void*>(y) && dtype != KVQ_DT_F32) return KVQ_ERR_INVALID_ARG;
  cudaError_t e = launch_tq4_rotate(*cache, x, dtype, y, rows, inverse ? 1 : 0, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

int32_t kvq_rotate_query(const void* x, int32_t dtype, float* y, int64_t rows, int32_t head_dim, void* stream) {
  if (rows < 0 || head_dim <= 0) return KVQ_ERR_INVALID_ARG;
  if (head_dim % 32 != 0) return KVQ_ERR_UNSUPPORTED;
  if (dtype != KVQ_DT_F32 && dtype != KVQ_DT_BF16) return KVQ_ERR_INVALID_ARG;
  if (rows == 0) return KVQ_OK;
  if (!x || !y) return KVQ_ERR_INVALID_ARG;
  if (x == static_cast<const void*>(y) && dtype != KVQ_DT_F32) return KVQ_ERR_INVALID_ARG;
  cudaError_t e = launch_rotate(x, dtype, y, rows, head_dim, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

int32_t kvq_store_rotate(const kvq_cache* cache, const void* k, const void* v, int32_t dtype, int64_t n_tok,
                         const int32_t* d_slot_mapping, int32_t* d_status, const void* q, int32_t q_dtype,
                         float* q_out, int64_t q_rows, void* stream) {
  int32_t st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_tok < 0 || q_rows < 0 || (dtype != KVQ_DT_F32 && dtype != KVQ_DT_BF16) ||
      (q_dtype != KVQ_DT_F32 && q_dtype != KVQ_DT_BF16))
    return KVQ_ERR_INVALID_ARG;
  if (!store_rotate_fits(*cache, n_tok)) return KVQ_ERR_UNSUPPORTED;
  if (n_tok > 0 && (!k || !v || !d_slot_mapping)) return KVQ_ERR_INVALID_ARG;
  if (q_rows > 0 && (!q || !q_out)) return KVQ_ERR_INVALID_ARG;
  if (q_rows > 0 && q == static_cast<const void*>(q_out) && q_dtype != KVQ_DT_F32) return KVQ_ERR_INVALID_ARG;
  cudaError_t e = launch_store_rotate(*cache, k, v, dtype, n_tok, d_slot_mapping, d_status, q, q_dtype, q_out, q_rows,
                                      cache->head_dim, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

size_t kvq_decode_workspace_size(const kvq_cache* cache, int32_t num_seqs, int32_t num_q_heads,
                                 int32_t max_seq_len, int32_t n_sel) {
  if (!cache || num_seqs < 0 || num_q_heads < 0 || max_seq_len < 0 || n_sel < 0 || cache->head_dim <= 0) return 0;
  return ws_layout(cache, num_seqs, num_q_heads, max_seq_len, n_sel).total;
}

static int32_t decode_attn_impl(const kvq_cache* cache, const float* q, const void* q_raw, int32_t q_dtype,
                                int32_t num_seqs, int32_t num_q_heads, const int32_t* d_seq_lens,
                                const int32_t* d_block_tables, int32_t max_pages_per_seq, int32_t max_seq_len,
                                const int32_t* d_sel, int32_t n_sel, float sm_scale, void* workspace, size_t ws_bytes,
                                void* stream, bool window = false, float* fused_out = nullptr,
                                const void* new_k = nullptr, const void* new_v = nullptr, int32_t new_dtype = 0) {
  int32_t st = check_cache(cache);
  if (st != KVQ_OK) return st;
  st = check_decode_shape(cache, num_seqs, num_q_heads, d_seq_lens, max_seq_len, d_sel != nullptr, n_sel);
  if (st != KVQ_OK) return st;
  if (num_seqs == 0) return KVQ_OK;
  if ((q_raw ? !aligned16(q_raw) : (!q || !aligned16(q))) || !d_block_tables || max_pages_per_seq < 1 || !workspace ||
      !aligned16(workspace))
    return KVQ_ERR_INVALID_ARG;
  if (!d_sel && static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_pages_per_seq) * cache->page_size)
    return KVQ_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(cache, num_seqs, num_q_heads, max_seq_len, d_sel ? n_sel : 0);
  if (ws_bytes < w.total) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int group = num_q_heads / cache->num_kv_heads;
  cudaError_t e;
  {
    const bool fp8 = cache->format == KVQ_FMT_FP8_ROW, bf16 = cache->format == KVQ_FMT_BF16;
    DecodeArgs a{};
    a.c = *cache;
    a.q = q;
    a.Hq = num_q_heads;
    a.group = group;
    a.seq_lens = d_seq_lens;
    a.block_tables = d_block_tables;
    a.max_pages = max_pages_per_seq;
    a.bt_stride = window ? 0 : max_pages_per_seq;
    a.nrows = window ? num_seqs : 0;
    a.max_seq_len = max_seq_len;
    a.sel = d_sel;
    a.n_sel = d_sel ? n_sel : 0;
    a.qscale = sm_scale * kLog2e;
    a.q_raw = q_raw;
    a.q_dtype = q_dtype;
    a.q_rotate = cache->format == KVQ_FMT_Q4_HAD32 ? 1 : 0;
    a.tq = cache->format == KVQ_FMT_TQ4 ? 1 : 0;
    a.ws_m = reinterpret_cast<float*>(ws + w.m_off);
    a.ws_z = reinterpret_cast<float*>(ws + w.z_off);
    a.ws_acc = reinterpret_cast<float*>(ws + w.acc_off);
    a.P = w.P;
    a.part = w.part;
    a.fused_out = fused_out;
    a.merge_ctr = reinterpret_cast<int32_t*>(ws + w.ctr_off);
    a.merge_B = num_seqs;
    a.merge_nblk = w.nblk;
    a.merge_m = reinterpret_cast<float*>(ws + w.bm_off);
    a.merge_z = reinterpret_cast<float*>(ws + w.bz_off);
    a.merge_acc = reinterpret_cast<float*>(ws + w.bacc_off);
    a.new_k = new_k;
    a.new_v = new_v;
    a.new_dtype = new_dtype;
    a.status = reinterpret_cast<int32_t*>(ws);
    // cache rows are 32-bit in the kernels (tensor-map coordinates, gathered row lists)
    const uint64_t rows = static_cast<uint64_t>(cache->num_pages) * cache->num_kv_heads * cache->page_size;
    if (rows >= (1ull << 31)) return KVQ_ERR_UNSUPPORTED;
    if (!d_sel) {
      bool ok;
      if (fp8)  // latent codes: 4 column boxes of 128 B; rope codes: one 64-byte box
        ok = encode_rows_map(&a.tm_k, cache->k, rows, 512, 16) &&
             encode_rows_map(&a.tm_v, cache->v, rows, 64, 16, 64, CU_TENSOR_MAP_SWIZZLE_64B);
      else if (bf16)  // 512-byte bf16 rows: 4 column boxes of 128 B
        ok = encode_rows_map(&a.tm_k, cache->k, rows, 512, 16) && encode_rows_map(&a.tm_v, cache->v, rows, 512, 16);
      else
        ok = encode_rows_map(&a.tm_k, cache->k, rows, 128, 16) && encode_rows_map(&a.tm_v, cache->v, rows, 128, 16);
      if (!ok) return cuda_fail(cudaErrorInvalidValue);
    }
    // An unrotated query on a grid of more than one wave: rotate it once, into
    // the block-partial area (only the fused merge uses it, and it holds at least
    // B x Hq x 256 floats), rather than in every CTA of every wave; the same
    // arithmetic, so the same bits
    if (q_raw && !fused_out && !decode_q4_one_wave(static_cast<int64_t>(w.P) * cache->num_kv_heads * num_seqs)) {
      if (a.q_rotate) {
        float* qr = reinterpret_cast<float*>(ws + w.bacc_off);
        e = launch_rotate(q_raw, q_dtype, qr, static_cast<int64_t>(num_seqs) * num_q_heads, cache->head_dim, s);
        if (e != cudaSuccess) return cuda_fail(e);
        a.q = qr;
        a.q_raw = nullptr;
      } else if (q_dtype == KVQ_DT_F32) {  // Q4_0 takes the query as given
        a.q = static_cast<const float*>(q_raw);
        a.q_raw = nullptr;
      }
    }
    e = fp8 ? launch_decode_fp8(a, num_seqs, s) : bf16 ? launch_decode_bf16(a, num_seqs, s) : launch_decode_q4(a, num_seqs, s);
  }
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

int32_t kvq_decode_attn(const kvq_cache* cache, const float* q, int32_t num_seqs, int32_t num_q_heads,
                        const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                        int32_t max_seq_len, const int32_t* d_sel, int32_t n_sel, float sm_scale, void* workspace,
                        size_t ws_bytes, void* stream) {
  return decode_attn_impl(cache, q, nullptr, 0, num_seqs, num_q_heads, d_seq_lens, d_block_tables,
                          max_pages_per_seq, max_seq_len, d_sel, n_sel, sm_scale, workspace, ws_bytes, stream);
}

int32_t kvq_decode_merged(const kvq_cache* cache, const float* q, int32_t num_seqs, int32_t num_q_heads,
                          const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                          int32_t max_seq_len, float sm_scale, void* workspace, size_t ws_bytes, float* out,
                          void* stream) {
  if (!cache) return KVQ_ERR_INVALID_ARG;
  if (!is_q4(cache->format)) return KVQ_ERR_UNSUPPORTED;
  if (num_seqs > 0 && !out) return KVQ_ERR_INVALID_ARG;
  // the last block folder keeps the group's block weights in its 32 KB of ring buffers
  const int64_t parts = (static_cast<int64_t>(max_seq_len) + kPart - 1) / kPart;
  const int64_t blocks = (parts + kMergeBlock - 1) / kMergeBlock;
  if (cache->num_kv_heads > 0 && num_q_heads > 0 && blocks * (num_q_heads / cache->num_kv_heads) > 8192)
    return KVQ_ERR_UNSUPPORTED;
  return decode_attn_impl(cache, q, nullptr, 0, num_seqs, num_q_heads, d_seq_lens, d_block_tables, max_pages_per_seq,
                          max_seq_len, nullptr, 0, sm_scale, workspace, ws_bytes, stream, false, out);
}

int32_t kvq_decode_window(const kvq_cache* cache, const float* q, int32_t num_rows, int32_t num_q_heads,
                          const int32_t* d_row_lens, const int32_t* d_block_table, int32_t max_pages,
                          int32_t max_seq_len, float sm_scale, void* workspace, size_t ws_bytes, void* stream) {
  if (!cache) return KVQ_ERR_INVALID_ARG;
  if (!is_q4(cache->format)) return KVQ_ERR_UNSUPPORTED;
  if (num_rows > 64) return KVQ_ERR_INVALID_ARG;
  return decode_attn_impl(cache, q, nullptr, 0, num_rows, num_q_heads, d_row_lens, d_block_table, max_pages,
                          max_seq_len, nullptr, 0, sm_scale, workspace, ws_bytes, stream, true);
}

int32_t kvq_decode_attn_unrotated(const kvq_cache* cache, const void* q, int32_t q_dtype, int32_t num_seqs,
                                  int32_t num_q_heads, const int32_t* d_seq_lens, const int32_t* d_block_tables,
                                  int32_t max_pages_per_seq, int32_t max_seq_len, const int32_t* d_sel,
                                  int32_t n_sel, float sm_scale, void* workspace, size_t ws_bytes, void* stream) {
  if (!cache || !is_q4(cache->format)) return cache ? KVQ_ERR_UNSUPPORTED : KVQ_ERR_INVALID_ARG;
  if (q_dtype != KVQ_DT_F32 && q_dtype != KVQ_DT_BF16) return KVQ_ERR_INVALID_ARG;
  if (num_seqs > 0 && !q) return KVQ_ERR_INVALID_ARG;
  return decode_attn_impl(cache, nullptr, q, q_dtype, num_seqs, num_q_heads, d_seq_lens, d_block_tables,
                          max_pages_per_seq, max_seq_len, d_sel, n_sel, sm_scale, workspace, ws_bytes, stream);
}

int32_t kvq_decode_step(const kvq_cache* cache, const void* k_new, const void* v_new, int32_t kv_dtype,
                        const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
                        const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                        int32_t max_seq_len, float sm_scale, void* workspace, size_t ws_bytes, void* stream) {
  if (!cache) return KVQ_ERR_INVALID_ARG;
  if (cache->format != KVQ_FMT_Q4_HAD32 && cache->format != KVQ_FMT_Q4_0) return KVQ_ERR_UNSUPPORTED;
  if ((kv_dtype != KVQ_DT_F32 && kv_dtype != KVQ_DT_BF16) || (q_dtype != KVQ_DT_F32 && q_dtype != KVQ_DT_BF16))
    return KVQ_ERR_INVALID_ARG;
  if (num_seqs > 0 && (!q || !k_new || !v_new)) return KVQ_ERR_INVALID_ARG;
  return decode_attn_impl(cache, nullptr, q, q_dtype, num_seqs, num_q_heads, d_seq_lens, d_block_tables,
                          max_pages_per_seq, max_seq_len, nullptr, 0, sm_scale, workspace, ws_bytes, stream, false,
                          nullptr, k_new, v_new, kv_dtype);
}

int32_t kvq_merge(const kvq_cache* cache, const void* workspace, size_t ws_bytes, int32_t num_seqs,
                  int32_t num_q_heads, const int32_t* d_seq_lens, int32_t max_seq_len, int32_t n_sel,
                  int32_t rotate_back, float* out, void* stream) {
  int32_t st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (n_sel < 0 || n_sel > 4096) return KVQ_ERR_INVALID_ARG;
  st = check_decode_shape(cache, num_seqs, num_q_heads, d_seq_lens, max_seq_len, n_sel > 0, n_sel);
  if (st != KVQ_OK) return st;
  if (rotate_back && cache->format != KVQ_FMT_Q4_HAD32 && cache->format != KVQ_FMT_TQ4) return KVQ_ERR_INVALID_ARG;
  if (num_seqs == 0) return KVQ_OK;
  if (!workspace || !out || !aligned16(workspace)) return KVQ_ERR_INVALID_ARG;
  const WsLayout w = ws_layout(cache, num_seqs, num_q_heads, max_seq_len, n_sel);
  if (ws_bytes < w.total) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  const uint8_t* ws = static_cast<const uint8_t*>(workspace);
  MergeArgs a{reinterpret_cast<const float*>(ws + w.m_off), reinterpret_cast<const float*>(ws + w.z_off),
              reinterpret_cast<const float*>(ws + w.acc_off), w.P, num_q_heads, value_width(cache), d_seq_lens,
              max_seq_len, n_sel, rotate_back && cache->format == KVQ_FMT_Q4_HAD32 ? 1 : 0, out, w.part};
  cudaError_t e = launch_merge(a, num_seqs, static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess && rotate_back && cache->format == KVQ_FMT_TQ4)  // the row transform needs the whole row
    e = launch_tq4_rotate(*cache, out, KVQ_DT_F32, out, static_cast<int64_t>(num_seqs) * num_q_heads, 1,
                          static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

int32_t kvq_prefill_attn(const kvq_cache* cache, const void* q, int32_t dtype, int32_t n_q, int32_t num_q_heads,
                         int32_t q_start, const int32_t* d_block_table, int32_t max_pages, float sm_scale, float* out,
                         int32_t* d_status, void* stream) {
  int32_t st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (!is_q4(cache->format) || cache->head_dim != 256) return KVQ_ERR_UNSUPPORTED;
  if (n_q < 0 || q_start < 0 || num_q_heads < 1 || num_q_heads % cache->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (dtype != KVQ_DT_F32 && dtype != KVQ_DT_BF16) return KVQ_ERR_INVALID_ARG;
  if (num_q_heads / cache->num_kv_heads > 8) return KVQ_ERR_UNSUPPORTED;
  if (n_q == 0) return KVQ_OK;
  if (!q || !out || !d_block_table || max_pages < 1) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(q_start) + n_q > static_cast<int64_t>(max_pages) * cache->page_size)
    return KVQ_ERR_INVALID_ARG;
  PrefillArgs a{};
  a.c = *cache;
  a.q = q;
  a.dtype = dtype;
  a.n_q = n_q;
  a.Hq = num_q_heads;
  a.group = num_q_heads / cache->num_kv_heads;
  a.q_start = q_start;
  a.block_table = d_block_table;
  a.max_pages = max_pages;
  a.qscale = sm_scale * kLog2e;
  a.out = out;
  a.status = d_status;
  a.rotate = cache->format == KVQ_FMT_Q4_HAD32 ? 1 : 0;
  {
    const uint64_t rows = static_cast<uint64_t>(cache->num_pages) * cache->num_kv_heads * cache->page_size;
    if (rows >= (1ull << 31)) return KVQ_ERR_UNSUPPORTED;
    if (!encode_rows_map(&a.tm_k, cache->k, rows, 128, 16) || !encode_rows_map(&a.tm_v, cache->v, rows, 128, 16))
      return cuda_fail(cudaErrorInvalidValue);
  }
  cudaError_t e = launch_prefill_tc(a, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

// fp8 streaming prefill: one partial (m, z, acc) per (row, head), the whole row
// being one partition.
static constexpr int kWholeRow = 1 << 30;

static WsLayout prefill_fp8_layout(int n_q, int Hq) {
  WsLayout w;
  w.P = 1;
  w.part = kWholeRow;
  const size_t n = static_cast<size_t>(n_q) * Hq;
  w.m_off = 256;
  w.z_off = w.m_off + round256(n * sizeof(float));
  w.acc_off = w.z_off + round256(n * sizeof(float));
  w.total = w.acc_off + round256(n * 512 * sizeof(float));
  return w;
}

size_t kvq_prefill_fp8_workspace_size(const kvq_cache* cache, int32_t n_q, int32_t num_q_heads) {
  if (!cache || n_q < 0 || num_q_heads < 0) return 0;
  return prefill_fp8_layout(n_q, num_q_heads).total;
}

int32_t kvq_prefill_attn_fp8(const kvq_cache* cache, const float* q, int32_t n_q, int32_t num_q_heads,
                             int32_t q_start, const int32_t* d_block_table, int32_t max_pages, float sm_scale,
                             void* workspace, size_t ws_bytes, float* out, void* stream) {
  int32_t st = check_cache(cache);
  if (st != KVQ_OK) return st;
  if (cache->format != KVQ_FMT_FP8_ROW) return KVQ_ERR_UNSUPPORTED;
  if (cache->head_dim != 512 || cache->rope_dim != 64 || num_q_heads < 16 || num_q_heads % 16 != 0)
    return KVQ_ERR_UNSUPPORTED;
  if (n_q < 0 || q_start < 0) return KVQ_ERR_INVALID_ARG;
  if (n_q == 0) return KVQ_OK;
  if (!q || !aligned16(q) || !out || !d_block_table || max_pages < 1 || !workspace || !aligned16(workspace))
    return KVQ_ERR_INVALID_ARG;
  const int64_t max_len = static_cast<int64_t>(q_start) + n_q;
  if (max_len > static_cast<int64_t>(max_pages) * cache->page_size || max_len >= kWholeRow) return KVQ_ERR_INVALID_ARG;
  const WsLayout w = prefill_fp8_layout(n_q, num_q_heads);
  if (ws_bytes < w.total) return KVQ_ERR_WORKSPACE_TOO_SMALL;
  const uint64_t rows = static_cast<uint64_t>(cache->num_pages) * cache->page_size;
  if (rows >= (1ull << 31)) return KVQ_ERR_UNSUPPORTED;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  DecodeArgs a{};
  a.c = *cache;
  a.q = q;
  a.Hq = num_q_heads;
  a.group = num_q_heads;
  a.block_tables = d_block_table;
  a.max_pages = max_pages;
  a.bt_stride = 0;  // every row reads the one table
  a.max_seq_len = static_cast<int>(max_len);
  a.qscale = sm_scale * kLog2e;
  a.ws_m = reinterpret_cast<float*>(ws + w.m_off);
  a.ws_z = reinterpret_cast<float*>(ws + w.z_off);
  a.ws_acc = reinterpret_cast<float*>(ws + w.acc_off);
  a.P = 1;
  a.part = w.part;
  a.status = reinterpret_cast<int32_t*>(ws);
  a.prefill = 1;
  a.prefill_q0 = q_start;
  if (!encode_rows_map(&a.tm_k, cache->k, rows, 512, 16) ||
      !encode_rows_map(&a.tm_v, cache->v, rows, 64, 16, 64, CU_TENSOR_MAP_SWIZZLE_64B))
    return cuda_fail(cudaErrorInvalidValue);
  cudaError_t e = launch_decode_fp8(a, n_q, s);
  if (e == cudaSuccess) {
    MergeArgs m{a.ws_m, a.ws_z, a.ws_acc, 1, num_q_heads, 512, nullptr, a.max_seq_len, 0, 0, out, w.part, 1, q_start};
    e = launch_merge(m, n_q, s);
  }
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

int32_t kvq_selftest_wait_timeout(int32_t* d_status, void* stream) {
  if (!d_status) return KVQ_ERR_INVALID_ARG;
  cudaError_t e = launch_wait_timeout_probe(d_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

int32_t kvq_read_status(const void* d_status, int32_t* host_code, void* stream) {
  if (!d_status || !host_code) return KVQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host_code, d_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  return e == cudaSuccess ? KVQ_OK : cuda_fail(e);
}

}  // extern "C"
