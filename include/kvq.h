/*
 * kvq.h -- C ABI of libkvq: attention over a sub-byte quantized KV cache on GB300.
 *
 * The library implements the hot path described on three public pages:
 *   [P1] "qwen27 CUDA: an opt-in 4-bit attention cache (262K on a 24 GB card)",
 *        section "What it is" -- rows of Hadamard-rotated 32-value groups kept as
 *        4-bit codes plus an fp16 scale (144 bytes for a 256-wide head); queries
 *        rotated once; attention in the rotated space over shared 512-key chunks
 *        plus the tail, merged in order; output rotated back once; prompt chunks
 *        packed into the cache and attended over decoded slots.
 *   [P2] "feat(kvcache): add reliable quantized KV cache", PR body -- 32 values
 *        -> 16 bytes + one fp16 scale; paged pools with a packed last dimension and
 *        a separate scale buffer; the engine rejects head_dim not divisible by 32.
 *   [P3] "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", KV8 base and
 *        split-T commits -- MLA latent rows as e4m3 with a per-row f32 scale
 *        amax/448; absorbed attention with (H,P) partials merged by log-sum-exp;
 *        a gather over selected absolute rows (at most 4096).
 *
 * Conventions for every entry point:
 *  - Pointers named d_* or documented as "device" are device pointers owned by the
 *    caller.  The library never allocates, frees or keeps device memory between
 *    calls; calls are reentrant and may come from several host threads.  (The one
 *    exception is kvq_decode_noalloc's fixed scratch array, described there.)
 *    Host-side state is limited to caches of per-call invariants, so that a call
 *    costs a launch and little more: the last 64 encoded TMA tensor maps (keyed
 *    by the plane's address and geometry, which is all a map holds; under a
 *    lock), each kernel's shared-memory attribute (set once per CUDA context)
 *    and the SM count per device.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work is
 *    enqueued asynchronously on it.
 *  - Host-side arguments are validated before anything is launched; on failure a
 *    negative kvq_status is returned and nothing is enqueued.  A failed launch
 *    returns KVQ_ERR_CUDA.
 *  - Device-resident metadata (slot mappings, block tables, sequence lengths,
 *    selected indices) cannot be checked on the host.  Kernels check it and, on a
 *    bad value, skip the access, write NaN to the affected output and OR a
 *    KVQ_DEV_* bit into the caller's status word; nothing traps.
 *  - Every kernel that waits (on a TMA copy) does so with an iteration limit and
 *    reports KVQ_DEV_TIMEOUT instead of hanging.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = -1,        /* null pointer, negative size, inconsistent shapes */
  KVQ_ERR_UNSUPPORTED = -2,        /* valid but not implemented (e.g. head_dim % 32 != 0) */
  KVQ_ERR_CUDA = -3,               /* a CUDA call failed; see kvq_last_cuda_error() */
  KVQ_ERR_WORKSPACE_TOO_SMALL = -4 /* ws_bytes < kvq_decode_workspace_size(...) */
} kvq_status;

/* Bits of the device status word (int32, caller-owned, zero it before use). */
enum {
  KVQ_DEV_BAD_SLOT = 1,      /* store: slot outside the pool */
  KVQ_DEV_BAD_PAGE = 2,      /* a block-table entry outside [0, num_pages) */
  KVQ_DEV_BAD_LENGTH = 4,    /* a sequence length < 0 or > the stated maximum */
  KVQ_DEV_BAD_INDEX = 8,     /* a selected index outside [0, seq_len) */
  KVQ_DEV_TIMEOUT = 16       /* a bounded wait on an asynchronous copy gave up */
};

/* Element type of caller-provided activations (new K/V rows, queries). */
typedef enum { KVQ_DT_F32 = 0, KVQ_DT_BF16 = 1 } kvq_dtype;

/* Cache formats.
 *
 * KVQ_FMT_Q4_HAD32 ([P1] "What it is"; [P2] PR body): every (position, KV head) row
 *   of head_dim D values is split into D/32 groups; each group is rotated by the
 *   orthonormal 32-point Walsh-Hadamard matrix H (natural Sylvester order,
 *   H[i][j] = (-1)^popcount(i&j) / sqrt(32)) and kept as 32 4-bit codes plus one
 *   fp16 scale:  scale = fp16_rne(amax/8) (saturated to 65504),
 *   code = clamp(rint_even(y / scale), -8, 7) + 8  (all codes 8 when scale == 0),
 *   value = (code - 8) * scale, in the rotated space.
 *   Codes plane: row r occupies D/2 bytes at r * D/2, the groups in order:
 *   group G at bytes 16G .. 16G + 15, byte b of it holding element 32G + 2b in
 *   the low nibble and 32G + 2b + 1 in the high nibble.
 *   Scale plane: row r occupies D/32 fp16 values at r * D/32, in group order.
 *   For D = 256 a row is 128 + 16 = 144 bytes.
 * KVQ_FMT_Q4_0 ([P2] PR body: 32 values -> 16 bytes + one fp16 scale, symmetric;
 *   the same shape as GGUF's Q4_0): KVQ_FMT_Q4_HAD32 without the rotation -- the
 *   same codes, scales and planes computed on the values as given.  Queries are
 *   used as given (kvq_rotate_query is not needed; kvq_decode_attn_unrotated and
 *   kvq_prefill_attn skip their rotations) and nothing is rotated back
 *   (kvq_merge with rotate_back = 0).
 * KVQ_FMT_TQ4 ([P3] "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", PR
 *   body, "Why rotated-int4": a randomized-Hadamard rotation and a fixed 16-level
 *   Lloyd-Max codebook for N(0,1) scaled by radius / sqrt(n), one scale per row):
 *   a row of D values (D = 64, 128 or 256) is signed by the cache's sign mask
 *   (bit i of signs[i / 32] set: element i negated), rotated by the D-point
 *   Walsh-Hadamard butterfly (stages h = 1 .. D/2, (a, b) -> (a + b, a - b),
 *   fp32) and multiplied by fp32(1/sqrt(D)); ss = the fp32 sum of the squares by
 *   the pairwise tree (stage h adds element i + h into i for i a multiple of
 *   2h); scale = fp16_rne(sqrtf(ss * (1/D))) (saturated to 65504); with
 *   v = y / scale (fp32 division) the code is 8 * [v < 0] + m, m = the number of
 *   midpoints (M_k + M_{k+1}) / 2, k < 7, below |v|, where M_0..M_7 =
 *   0.12841796875, 0.387939453125, 0.65673828125, 0.9423828125, 1.255859375,
 *   1.6181640625, 2.068359375, 2.732421875 (the Lloyd-Max levels rounded to
 *   fp16); scale 0 stores code 0.  value = (code & 8 ? -1 : 1) * M_{code & 7} *
 *   scale, in the rotated space.  Codes plane as for KVQ_FMT_Q4_HAD32 (element
 *   2b of the row in the low nibble of byte b); scale plane: one fp16 per row.
 *   For D = 256 a row is 128 + 2 = 130 bytes.  Queries are rotated by the same
 *   signed transform (kvq_tq4_rotate) and outputs rotated back by its inverse
 *   (kvq_merge with rotate_back, or kvq_tq4_rotate with inverse = 1).
 * KVQ_FMT_BF16: unrotated bf16 rows of D values (the uncompressed comparison).
 * KVQ_FMT_FP8_ROW ([P3] KV8 base commit): one latent row per position (num_kv_heads
 *   must be 1): head_dim latent values ("Lc") and rope_dim rope values ("Rc"), each
 *   part kept as e4m3 bytes with its own f32 scale amax/448: inv = 448/amax (fp32),
 *   code = e4m3_rne_satfinite(x * inv); amax == 0 or a non-finite inv stores zero
 *   codes; NaN inputs store 0x00.  In attention the key is Lc ++ Rc and the value
 *   is Lc (absorbed attention: the latent is both key and value).
 *
 * Row index of (page, kv_head, slot) in every plane:
 *   r = (page * num_kv_heads + kv_head) * page_size + slot.
 * A token's slot number is page * page_size + slot; block tables list page ids. */
typedef enum {
  KVQ_FMT_Q4_HAD32 = 0,
  KVQ_FMT_BF16 = 1,
  KVQ_FMT_FP8_ROW = 2,
  KVQ_FMT_Q4_0 = 3,
  KVQ_FMT_TQ4 = 4
} kvq_format;

typedef struct kvq_cache {
  int32_t format;       /* kvq_format */
  int32_t num_kv_heads; /* Hk (FP8_ROW: 1) */
  int32_t head_dim;     /* D: key/value width (FP8_ROW: latent width) */
  int32_t rope_dim;     /* FP8_ROW: rope width; otherwise 0 */
  int32_t page_size;    /* slots per page; a positive multiple of 16 */
  int32_t num_pages;    /* pages in the pool */
  void* k;              /* Q4: K codes plane (u8); BF16: K plane; FP8_ROW: Lc codes [rows][D] */
  void* k_scale;        /* Q4: K scale plane (fp16); BF16: unused; FP8_ROW: Lc scales [rows] f32 */
  void* v;              /* Q4: V codes plane; BF16: V plane; FP8_ROW: Rc codes [rows][rope_dim] */
  void* v_scale;        /* Q4: V scale plane; BF16: unused; FP8_ROW: Rc scales [rows] f32 */
  const void* signs;    /* TQ4: device uint32 [head_dim / 32], the rotation's sign mask; otherwise unused */
} kvq_cache;

/* Version of the ABI (major * 10000 + minor * 100 + patch). */
int32_t kvq_version(void);
/* Short text of a kvq_status value (static storage). */
const char* kvq_status_string(int32_t status);
/* The cudaError_t of the last KVQ_ERR_CUDA returned on this thread (0 if none). */
int32_t kvq_last_cuda_error(void);

/* Bytes of each plane for a cache description (0 for unused planes). */
size_t kvq_plane_bytes(const kvq_cache* cache, int32_t plane /* 0 k, 1 k_scale, 2 v, 3 v_scale */);

/* kvq_store -- pack new tokens into the cache ([P1] "What it is": "pack the
 * window's new keys and values the same way"; [P3] KV8 base: the producer
 * quantises the fresh row).
 *   k, v:   device, [n_tok, num_kv_heads, head_dim] of dtype (Q4 / BF16).
 *           FP8_ROW: k is [n_tok, head_dim + rope_dim] and v must be NULL.
 *   d_slot_mapping: device int32 [n_tok]; slot = page * page_size + offset;
 *           a negative slot skips the token; a slot >= num_pages * page_size is
 *           skipped and flagged KVQ_DEV_BAD_SLOT.
 *   d_status: optional device int32 status word (may be NULL).
 * Bit-exact with the definition above (fp32 rotation by the butterfly with
 * stages 1, 2, 4, 8, 16, then one multiply by fp32(1/sqrt(32)); IEEE division;
 * round half to even).  Rows are independent: storing tokens one by one or all
 * at once writes the same bytes. */
int32_t kvq_store(const kvq_cache* cache, const void* k, const void* v, int32_t dtype, int64_t n_tok,
                  const int32_t* d_slot_mapping, int32_t* d_status, void* stream);

/* kvq_rotate_query -- y = blockdiag(H) x for `rows` rows of head_dim values
 * ([P1] "What it is": rotate the queries once; H is its own inverse, so the same
 * call rotates an output back).  x: device [rows, head_dim] of dtype; y: device
 * fp32 [rows, head_dim]; y may equal x when dtype is F32.  head_dim % 32 == 0. */
int32_t kvq_rotate_query(const void* x, int32_t dtype, float* y, int64_t rows, int32_t head_dim,
                         void* stream);

/* kvq_tq4_rotate -- the TQ4 format's rotation of `rows` rows of head_dim values:
 * inverse = 0: y = H (s * x) / sqrt(D) (queries into the cache's space);
 * inverse = 1: y = s * (H x) / sqrt(D) (outputs back), s the cache's signs, H
 * the D-point Walsh-Hadamard matrix ([P3] "Why rotated-int4": randomized
 * Hadamard).  fp32 butterfly; x: device [rows, head_dim] of dtype; y: device
 * fp32 [rows, head_dim], may equal x when dtype is F32.  KVQ_ERR_UNSUPPORTED for
 * a cache of another format. */
int32_t kvq_tq4_rotate(const kvq_cache* cache, const void* x, int32_t dtype, float* y, int64_t rows,
                       int32_t inverse, void* stream);

/* kvq_store_rotate -- kvq_store of n_tok new tokens and kvq_rotate_query of
 * q_rows query rows (of the cache's head_dim) in one launch.  A decode step's
 * two preparations are independent of each other ([P1] "What it is": pack the
 * new keys and values; rotate the queries once), so one kernel does both and
 * the step pays one launch latency instead of two.  Same bytes and the same
 * rotated values as the two calls.  Arguments as for kvq_store (4-bit format
 * only) and kvq_rotate_query (q: [q_rows, head_dim] of q_dtype; q_out: fp32;
 * q_out may equal q when q_dtype is F32).  Only for the few-row form of the
 * store (n_tok * num_kv_heads * 2 <= 256, head_dim in {32, 64, 128, 256});
 * otherwise KVQ_ERR_UNSUPPORTED (make the two calls). */
int32_t kvq_store_rotate(const kvq_cache* cache, const void* k, const void* v, int32_t dtype, int64_t n_tok,
                         const int32_t* d_slot_mapping, int32_t* d_status, const void* q, int32_t q_dtype,
                         float* q_out, int64_t q_rows, void* stream);

/* Size in bytes of the workspace kvq_decode_attn needs for this problem:
 * a 256-byte header (status word at offset 0), then partial maxima m and sums z
 * [num_seqs][num_q_heads][P] f32 and partial contexts acc [num_seqs][num_q_heads]
 * [P][value width] f32, where P = ceil(max_seq_len / 512), or for a gather
 * P = ceil(n_sel / 512) (FP8_ROW: ceil(n_sel / 64)); then kvq_decode_merged's
 * completion counters, int32 [num_seqs][num_kv_heads] and [num_seqs]
 * [num_kv_heads][ceil(P / 8)] (zero before the first kvq_decode_merged on the
 * workspace; each complete call leaves them zero), and its block partials
 * (m, z [num_seqs][num_q_heads][ceil(P / 8)] f32, acc [..][value width] f32). */
size_t kvq_decode_workspace_size(const kvq_cache* cache, int32_t num_seqs, int32_t num_q_heads,
                                 int32_t max_seq_len, int32_t n_sel);

/* kvq_decode_attn -- split-T decode attention partials ([P1] "What it is": attend
 * over the 4-bit cache in rotated space over shared 512-key chunks plus the tail;
 * [P3] split-T commit: dim3(H,P) partial online-softmax blocks (cl, m, z)).
 * For sequence b, query head h (reading KV head h / (num_q_heads / num_kv_heads))
 * and partition p (keys [512p, min(512p + 512, T_b)), T_b = seq_lens[b], or the
 * p-th run of 512 entries of sel[b] when gathering -- 64 entries for FP8_ROW),
 * writes
 *   m = max_j s_j * log2(e),  z = sum_j 2^(s_j log2(e) - m),
 *   acc = sum_j 2^(s_j log2(e) - m) * value_j,   s_j = sm_scale * (q . key_j)
 * into the workspace.  Empty partitions get m = -inf, z = 0, acc = 0.
 *   q:  device fp32 [num_seqs, num_q_heads, key width]; Q4: already rotated
 *       (kvq_rotate_query); TQ4: already rotated (kvq_tq4_rotate); BF16 /
 *       FP8_ROW: as is.  Key width = head_dim (+ rope_dim for FP8_ROW).
 *   d_seq_lens: device int32 [num_seqs], each in [0, max_seq_len].
 *   d_block_tables: device int32 [num_seqs, max_pages_per_seq].
 *   d_sel: NULL for dense attention, else device int32 [num_seqs, n_sel] absolute
 *       positions, each < seq_lens[b] (gather; n_sel <= 4096, [P3] split-T commit).
 *   Q4 / TQ4 / BF16 need num_q_heads / num_kv_heads <= 8 and head_dim == 256
 *   (TQ4: dense only, d_sel must be NULL).
 *   FP8_ROW needs head_dim == 512, rope_dim == 64 and num_q_heads % 16 == 0. */
int32_t kvq_decode_attn(const kvq_cache* cache, const float* q, int32_t num_seqs, int32_t num_q_heads,
                        const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                        int32_t max_seq_len, const int32_t* d_sel, int32_t n_sel, float sm_scale,
                        void* workspace, size_t ws_bytes, void* stream);

/* kvq_decode_window -- kvq_decode_attn for a window of num_rows query rows of ONE
 * sequence that share its block table: the draft rows of a speculative-decoding
 * step ([P1] "What it is": shared 512-key chunks plus each row's causal tail).
 * Row i attends keys 0 .. d_row_lens[i] - 1 of the sequence (a causal window:
 * prefix_len + i + 1; the lengths may come in any order).  One pass over each
 * 512-key partition serves every row: the (row, head) pairs of up to
 * floor(32 / group) rows face the keys together (more rows are cut into even
 * slices), so a key's codes are read once and converted once for all of them,
 * and each row masks the keys past its own end.  The partials are bit-identical
 * to kvq_decode_attn with num_seqs = num_rows, seq_lens = d_row_lens and the
 * block table repeated for every row.  A row whose length is out of range is
 * skipped and flagged (KVQ_DEV_BAD_LENGTH; the merge writes NaN for it), the
 * others are unaffected.
 * Merge with kvq_merge(num_seqs = num_rows, d_seq_lens = d_row_lens).
 *   q: device fp32 [num_rows, num_q_heads, head_dim] (rotated, as for
 *      kvq_decode_attn); d_row_lens: device int32 [num_rows];
 *   d_block_table: device int32 [max_pages], shared by every row.
 *   4-bit formats only (else KVQ_ERR_UNSUPPORTED); 1 <= num_rows <= 64.
 * Workspace (kvq_decode_workspace_size with num_seqs = num_rows) and errors as
 * for kvq_decode_attn. */
int32_t kvq_decode_window(const kvq_cache* cache, const float* q, int32_t num_rows, int32_t num_q_heads,
                          const int32_t* d_row_lens, const int32_t* d_block_table, int32_t max_pages,
                          int32_t max_seq_len, float sm_scale, void* workspace, size_t ws_bytes, void* stream);

/* kvq_decode_step -- one decode step of a 4-bit cache in one launch: each
 * sequence appends its new token and attends with its query ([P1] "What it is":
 * pack the new keys and values, then attend over the 4-bit cache).  For sequence
 * b the new rows k_new[b], v_new[b] are stored at logical position
 * seq_lens[b] - 1 (the cache row d_block_tables maps it to) exactly as kvq_store
 * stores them, the query q[b] is rotated exactly as kvq_rotate_query rotates it
 * (KVQ_FMT_Q4_HAD32; KVQ_FMT_Q4_0 uses it as given), and the partials are those
 * of kvq_decode_attn over positions [0, seq_lens[b]): the same bits as
 * kvq_store + kvq_rotate_query + kvq_decode_attn.  Inside the launch, the CTA of
 * each (sequence, KV head) whose 512-key partition holds the new position writes
 * the token before it reads its tiles; no other CTA reads that row.  A grid of
 * more than one wave (over two CTAs per SM) of a KVQ_FMT_Q4_HAD32 cache takes a
 * second launch first that rotates the queries once into the workspace (the
 * in-kernel rotation would be repeated by every CTA of every wave); a KVQ_FMT_Q4_0
 * cache with fp32 queries then reads q as given.  Merge with kvq_merge.
 *   k_new, v_new: device [num_seqs, num_kv_heads, head_dim] of kv_dtype;
 *   q: device [num_seqs, num_q_heads, head_dim] of q_dtype, not rotated.
 *   A sequence of length 0 stores nothing (its outputs are zeros); a new
 *   position whose block-table entry is outside the pool stores nothing and the
 *   decode flags KVQ_DEV_BAD_PAGE as kvq_decode_attn does.
 * KVQ_FMT_Q4_HAD32 and KVQ_FMT_Q4_0 only (else KVQ_ERR_UNSUPPORTED); head_dim
 * 256.  Workspace (kvq_decode_workspace_size with n_sel = 0) and errors as for
 * kvq_decode_attn. */
int32_t kvq_decode_step(const kvq_cache* cache, const void* k_new, const void* v_new, int32_t kv_dtype,
                        const void* q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
                        const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                        int32_t max_seq_len, float sm_scale, void* workspace, size_t ws_bytes, void* stream);

/* kvq_decode_merged -- kvq_decode_attn and kvq_merge (with the rotation back for
 * Q4_HAD32) in one launch ([P1] "What it is": the shared 512-key chunks and the
 * in-order merge of one decode round).  The merge runs in two levels inside the
 * decode kernel: the last CTA to finish among each block of 8 consecutive
 * partitions of a (sequence, KV head) folds that block's partials (ascending
 * partition order) into a block partial, and the last block folder of the
 * (sequence, KV head) folds the block partials (ascending) and writes out
 * [num_seqs, num_q_heads, 256] fp32.  The tree depends only on the partition
 * indices, so the values do not depend on the batch or on the order in which
 * CTAs finish; they equal kvq_merge's up to the grouping of the fp32 sums.
 *   Arguments as for kvq_decode_attn (dense; 4-bit formats, else
 *   KVQ_ERR_UNSUPPORTED); ceil(ceil(max_seq_len / 512) / 8) * (num_q_heads /
 *   num_kv_heads) <= 8192.  An invalid length gives NaN rows (and
 *   KVQ_DEV_BAD_LENGTH), an empty sequence zeros. */
int32_t kvq_decode_merged(const kvq_cache* cache, const float* q, int32_t num_seqs, int32_t num_q_heads,
                          const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                          int32_t max_seq_len, float sm_scale, void* workspace, size_t ws_bytes, float* out,
                          void* stream);

/* kvq_decode_attn_unrotated -- kvq_decode_attn for the 4-bit format with the
 * query rotation done inside the decode kernel ([P1] "What it is": the query
 * is rotated once, then the 4-bit cache is streamed in rotated space), saving the
 * separate kvq_rotate_query launch of a decode step.  Every CTA (one per 512-key
 * partition and KV head) repeats the rotation of its group's queries, which
 * pays off while the grid runs in one wave (up to two CTAs per SM); a larger
 * grid (it measured +6 us per layer at 262K keys) takes a rotation launch first
 * instead, into the workspace, as kvq_decode_step does.
 *   q: device [num_seqs, num_q_heads, 256] of q_dtype (KVQ_DT_F32 or KVQ_DT_BF16),
 *      unrotated (KVQ_FMT_Q4_0: used as given).  The queries of each GQA group
 *      are rotated with the arithmetic of kvq_rotate_query, so the partials
 *      equal those of kvq_rotate_query + kvq_decode_attn bit for bit.
 * Other arguments, workspace and errors as for kvq_decode_attn; formats other
 * than Q4_HAD32 and Q4_0 return KVQ_ERR_UNSUPPORTED. */
int32_t kvq_decode_attn_unrotated(const kvq_cache* cache, const void* q, int32_t q_dtype, int32_t num_seqs,
                                  int32_t num_q_heads, const int32_t* d_seq_lens, const int32_t* d_block_tables,
                                  int32_t max_pages_per_seq, int32_t max_seq_len, const int32_t* d_sel,
                                  int32_t n_sel, float sm_scale, void* workspace, size_t ws_bytes, void* stream);

/* kvq_merge -- log-sum-exp merge of the partials ([P1] "in-order merge ... and
 * rotate the output back once"; [P3] split-T commit: merge kernel):
 *   M = max_p m_p,  Z = sum_p z_p 2^(m_p - M),  o = sum_p acc_p 2^(m_p - M) / Z,
 * taking partitions in ascending order in a fixed grouping (runs are
 * bit-reproducible), then out = blockdiag(H) o when rotate_back != 0 (Q4_HAD32),
 * or out = s * (H o) / sqrt(D) (TQ4: a second launch on out; the other formats
 * take rotate_back = 0).
 * A sequence with no keys gives zeros.  Arguments as for kvq_decode_attn.
 * out: device fp32 [num_seqs, num_q_heads, value width]. */
int32_t kvq_merge(const kvq_cache* cache, const void* workspace, size_t ws_bytes, int32_t num_seqs,
                  int32_t num_q_heads, const int32_t* d_seq_lens, int32_t max_seq_len, int32_t n_sel,
                  int32_t rotate_back, float* out, void* stream);

/* kvq_prefill_attn -- causal attention of a prompt chunk over decoded slots
 * ([P1] "What it is": prompt chunks are packed into the cache, then attended with
 * the prefill-attention kernel over decoded slots).  Query i (absolute position
 * q_start + i) attends keys 0 .. q_start + i of the sequence whose block table is
 * d_block_table; the chunk's own keys must already be stored (kvq_store).
 *   q:   device [n_q, num_q_heads, head_dim] of dtype, unrotated.
 *   out: device fp32 [n_q, num_q_heads, head_dim], rotated back.
 *   Q4 only; head_dim == 256; num_q_heads / num_kv_heads <= 8. */
int32_t kvq_prefill_attn(const kvq_cache* cache, const void* q, int32_t dtype, int32_t n_q,
                         int32_t num_q_heads, int32_t q_start, const int32_t* d_block_table,
                         int32_t max_pages, float sm_scale, float* out, int32_t* d_status, void* stream);

/* Size in bytes of the workspace kvq_prefill_attn_fp8 needs: a 256-byte header
 * (status word at offset 0), then m, z [n_q][num_q_heads] f32 and acc
 * [n_q][num_q_heads][512] f32 (one partial per row and head). */
size_t kvq_prefill_fp8_workspace_size(const kvq_cache* cache, int32_t n_q, int32_t num_q_heads);

/* kvq_prefill_attn_fp8 -- causal attention of a prompt chunk over the fp8
 * latent cache ([P3] "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant",
 * split-T commit: the batch / prefill path keeps a tiled streaming kernel with
 * one block per (row, heads), the length cap lifted to 1M): query i (absolute
 * position q_start + i) attends keys 0 .. q_start + i, absorbed as in
 * kvq_decode_attn (key = Lc ++ Rc, value = Lc).  One CTA per (block of 32
 * heads, row) streams all of the row's keys with an online softmax (the row is
 * one partition), then the merge normalises; no length cap beyond the cache.
 *   q: device fp32 [n_q, num_q_heads, 576]; out: device fp32 [n_q, num_q_heads, 512].
 *   d_block_table: device int32 [max_pages], the chunk's sequence;
 *   q_start + n_q <= max_pages * page_size.
 *   FP8_ROW only (head_dim 512, rope_dim 64, num_q_heads % 16 == 0), else
 *   KVQ_ERR_UNSUPPORTED.  Bad pages are flagged in the workspace's status word
 *   (KVQ_DEV_BAD_PAGE) and the affected rows come out NaN. */
int32_t kvq_prefill_attn_fp8(const kvq_cache* cache, const float* q, int32_t n_q, int32_t num_q_heads,
                             int32_t q_start, const int32_t* d_block_table, int32_t max_pages, float sm_scale,
                             void* workspace, size_t ws_bytes, float* out, void* stream);

/* Copy the device status word at the start of a decode workspace (or any
 * device int32) to *host_code; synchronises `stream`. */
int32_t kvq_read_status(const void* d_status, int32_t* host_code, void* stream);

/* kvq_selftest_wait_timeout -- diagnostic of the kernels' copy waits: one CTA
 * waits on a shared-memory barrier that nothing completes, with the same bounded
 * wait the kernels use (about 2 seconds), and ORs KVQ_DEV_TIMEOUT into
 * *d_status when it gives up.  The kernel then returns normally, so the CUDA
 * context stays usable.  d_status: device int32. */
int32_t kvq_selftest_wait_timeout(int32_t* d_status, void* stream);

/* kvq_decode_noalloc -- kvq_decode_attn followed by kvq_merge, for callers that
 * cannot allocate device memory when they decode (a host that owns every device
 * allocation, a memory pool that forbids new ones, a latency-critical path that
 * cannot afford cudaMalloc).  The pages have no counterpart: this is an
 * interface convenience of this library, with the same arithmetic (and the same
 * output bits) as the two calls it replaces.
 * Instead of a caller workspace it uses one file-scope device array of
 * kvq_noalloc_scratch_bytes() bytes (16 MiB), which every GPU that loads the
 * library holds until the process exits.  Problems whose workspace
 * (kvq_decode_workspace_size) exceeds it are rejected with
 * KVQ_ERR_WORKSPACE_TOO_SMALL.  Every argument check of the two calls runs
 * before anything is enqueued; an invalid call enqueues nothing.
 * Set-up: the array's device address is looked up (cudaGetSymbolAddress, with
 * the device current) on the first call in each CUDA context and cached with
 * that context's ID; a call in another context (a non-primary context made
 * current by the caller, or the primary context re-created after
 * cudaDeviceReset) looks it up again.  The library loads its modules lazily, so
 * that first call also loads the array's module and commits its 16 MiB of
 * device memory: make it outside any region where the caller cannot allocate,
 * and before any stream capture.  Later calls allocate and free nothing.
 * All calls share the array and it keeps the last call's contents; the status
 * word is cleared on `stream` at the start of every call.  Calls whose GPU work
 * overlaps (on different streams without ordering) race on the array.
 * Arguments as for kvq_decode_attn and kvq_merge; d_status_out (optional device
 * int32) receives a copy of the call's status word. */
size_t kvq_noalloc_scratch_bytes(void);
int32_t kvq_decode_noalloc(const kvq_cache* cache, const float* q, int32_t num_seqs, int32_t num_q_heads,
                           const int32_t* d_seq_lens, const int32_t* d_block_tables, int32_t max_pages_per_seq,
                           int32_t max_seq_len, const int32_t* d_sel, int32_t n_sel, float sm_scale,
                           int32_t rotate_back, float* out, int32_t* d_status_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* KVQ_H */
