// store.cu -- packing new rows into the cache, and the query rotation.
//
// kvq_store for the rotated 4-bit format follows "qwen27 CUDA: an opt-in 4-bit
// attention cache (262K on a 24 GB card)", section "What it is" (Hadamard-rotated
// groups of 32 values as 4-bit codes plus an fp16 scale) and "feat(kvcache): add
// reliable quantized KV cache", PR body (32 values -> 16 bytes + one fp16 scale,
// symmetric codes).  The fp8 latent rows follow "KV cache quantization: fp8
// (KV8) + 4-bit TurboQuant", KV8 base commit (e4m3 bytes, per-row f32 scale
// amax/448, RNE encoder saturating at +-448, NaN stored as 0, guard for a
// subnormal amax).
//
// This translation unit is compiled with -fmad=false: every operation below is
// a single IEEE-rounded fp32 operation, so the codes are bit-exact with the
// definition in kvq.h.
#include <cuda_fp8.h>

#include "kernels.cuh"

namespace kvq {

// One warp per (token, KV head, K|V) row of D = 32*NG values.
// Lane i handles element 32G + i of every group G.  ROT = false: the unrotated
// Q4_0 format (the values as given).
template <int NG, bool ROT>
__global__ void __launch_bounds__(256) store_q4_kernel(kvq_cache c, const void* __restrict__ k,
                                                       const void* __restrict__ v, int dtype, int64_t n_tok,
                                                       const int32_t* __restrict__ slots, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  constexpr int D = NG * 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int Hk = c.num_kv_heads;
  if (row >= n_tok * Hk * 2) return;
  const int kv = static_cast<int>(row & 1);
  const int64_t tok = (row >> 1) / Hk;
  const int head = static_cast<int>((row >> 1) % Hk);
  const int32_t slot = slots[tok];
  if (slot < 0) return;
  if ((int64_t)slot >= (int64_t)c.num_pages * c.page_size) {
    if (lane == 0) set_status(status, KVQ_DEV_BAD_SLOT);
    return;
  }
  const int64_t page = slot / c.page_size;
  const int off = slot % c.page_size;
  const int64_t r = (page * Hk + head) * c.page_size + off;
  const void* src = kv ? v : k;
  const int64_t base = (tok * Hk + head) * D;

  // The warp's row is staged in shared memory (group G's 16 bytes at 16G) and
  // then written with one 16-byte store per group.
  __shared__ __align__(16) uint8_t stage[8][NG * 16];
  uint8_t* my_stage = stage[threadIdx.x >> 5];
  uint16_t scale16[NG];  // warp-uniform
#pragma unroll
  for (int G = 0; G < NG; ++G) {
    float x = load_act(src, dtype, base + 32 * G + lane);
    const float y = ROT ? __fmul_rn(warp_fwht32(x, lane), kHadamardScale) : x;
    float amax = fabsf(y);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s32 = __fdiv_rn(amax, 8.0f);
    __half s16 = __float2half_rn(s32);
    if (__hisinf(s16)) s16 = __ushort_as_half(0x7BFFu);  // saturate to 65504
    const float s = __half2float(s16);
    int code = 8;
    if (s != 0.0f) {
      float q = rintf(__fdiv_rn(y, s));
      q = fminf(fmaxf(q, -8.0f), 7.0f);
      code = static_cast<int>(q) + 8;
    }
    // gather the four codes of half-word h = lane/4 (elements 4h .. 4h+3) into lane 4h
    uint32_t bits = static_cast<uint32_t>(code) << (4 * (lane & 3));
    bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
    bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
    if ((lane & 3) == 0) reinterpret_cast<uint16_t*>(my_stage)[8 * G + (lane >> 2)] = static_cast<uint16_t>(bits);
    scale16[G] = __half_as_ushort(s16);
  }
  __syncwarp();
  uint8_t* codes = static_cast<uint8_t*>(kv ? c.v : c.k) + r * (D / 2);
  if (lane < NG) reinterpret_cast<uint4*>(codes)[lane] = reinterpret_cast<const uint4*>(my_stage)[lane];
  uint16_t* sc = static_cast<uint16_t*>(kv ? c.v_scale : c.k_scale) + r * NG;
  if (lane < NG) {
    uint16_t mine = 0;
#pragma unroll
    for (int G = 0; G < NG; ++G)
      if (G == lane) mine = scale16[G];
    sc[lane] = mine;
  }
}

// Latency form of the same store for a handful of rows (a decode step stores one
// token): one warp per (row, group), so the groups of a row are packed in
// parallel instead of one after another.  Same arithmetic, same bytes.
// Warp `wid` of the store: (row, group) = (wid / NG, wid % NG).
template <int NG, bool ROT>
__device__ __forceinline__ void store_q4_group_warp(const kvq_cache& c, const void* __restrict__ k,
                                                    const void* __restrict__ v, int dtype, int64_t n_tok,
                                                    const int32_t* __restrict__ slots, int32_t* status, int64_t wid) {
  constexpr int D = NG * 32;
  const int lane = threadIdx.x & 31;
  const int Hk = c.num_kv_heads;
  if (wid >= n_tok * Hk * 2 * NG) return;
  const int G = static_cast<int>(wid % NG);
  const int64_t row = wid / NG;
  const int kv = static_cast<int>(row & 1);
  const int64_t tok = (row >> 1) / Hk;
  const int head = static_cast<int>((row >> 1) % Hk);
  const int32_t slot = slots[tok];
  if (slot < 0) return;
  if ((int64_t)slot >= (int64_t)c.num_pages * c.page_size) {
    if (lane == 0 && G == 0) set_status(status, KVQ_DEV_BAD_SLOT);
    return;
  }
  const int64_t page = slot / c.page_size;
  const int off = slot % c.page_size;
  const int64_t r = (page * Hk + head) * c.page_size + off;
  const void* src = kv ? v : k;
  float x = load_act(src, dtype, (tok * Hk + head) * D + 32 * G + lane);
  const float y = ROT ? __fmul_rn(warp_fwht32(x, lane), kHadamardScale) : x;
  float amax = fabsf(y);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s32 = __fdiv_rn(amax, 8.0f);
  __half s16 = __float2half_rn(s32);
  if (__hisinf(s16)) s16 = __ushort_as_half(0x7BFFu);  // saturate to 65504
  const float s = __half2float(s16);
  int code = 8;
  if (s != 0.0f) {
    float q = rintf(__fdiv_rn(y, s));
    q = fminf(fmaxf(q, -8.0f), 7.0f);
    code = static_cast<int>(q) + 8;
  }
  uint32_t bits = static_cast<uint32_t>(code) << (4 * (lane & 3));
  bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
  bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
  uint8_t* codes = static_cast<uint8_t*>(kv ? c.v : c.k) + r * (D / 2);
  if ((lane & 3) == 0) {
    const int h = lane >> 2;  // half-word h of group G: bytes 16G + 2h, 16G + 2h + 1
    reinterpret_cast<uint16_t*>(codes)[8 * G + h] = static_cast<uint16_t>(bits);
  }
  if (lane == 0) (static_cast<uint16_t*>(kv ? c.v_scale : c.k_scale) + r * NG)[G] = __half_as_ushort(s16);
}

template <int NG, bool ROT>
__global__ void __launch_bounds__(256) store_q4_group_kernel(kvq_cache c, const void* __restrict__ k,
                                                             const void* __restrict__ v, int dtype, int64_t n_tok,
                                                             const int32_t* __restrict__ slots, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  store_q4_group_warp<NG, ROT>(c, k, v, dtype, n_tok, slots, status,
                               (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
}

// BF16 comparison format: plain copy / RNE conversion of each value.
__global__ void store_bf16_kernel(kvq_cache c, const void* __restrict__ k, const void* __restrict__ v, int dtype,
                                  int64_t n_tok, const int32_t* __restrict__ slots, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int D = c.head_dim, Hk = c.num_kv_heads;
  const int64_t total = n_tok * Hk * D;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = i / ((int64_t)Hk * D);
    const int head = static_cast<int>((i / D) % Hk);
    const int d = static_cast<int>(i % D);
    const int32_t slot = slots[tok];
    if (slot < 0) continue;
    if ((int64_t)slot >= (int64_t)c.num_pages * c.page_size) {
      if (d == 0 && head == 0) set_status(status, KVQ_DEV_BAD_SLOT);
      continue;
    }
    const int64_t r = ((int64_t)(slot / c.page_size) * Hk + head) * c.page_size + slot % c.page_size;
    __nv_bfloat16* kd = static_cast<__nv_bfloat16*>(c.k) + r * D + d;
    __nv_bfloat16* vd = static_cast<__nv_bfloat16*>(c.v) + r * D + d;
    if (dtype == KVQ_DT_BF16) {
      *kd = static_cast<const __nv_bfloat16*>(k)[i];
      *vd = static_cast<const __nv_bfloat16*>(v)[i];
    } else {
      *kd = __float2bfloat16_rn(static_cast<const float*>(k)[i]);
      *vd = __float2bfloat16_rn(static_cast<const float*>(v)[i]);
    }
  }
}

__device__ __forceinline__ uint8_t e4m3_encode(float x) {
  if (isnan(x)) return 0;  // NaN is stored as the inert code 0
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// One block (128 threads) per token: latent part and rope part each get amax,
// inv = 448/amax (fp32), codes e4m3(x * inv), scale amax/448.
__global__ void __launch_bounds__(128) store_fp8_kernel(kvq_cache c, const void* __restrict__ rows, int dtype,
                                                         int64_t n_tok, const int32_t* __restrict__ slots,
                                                         int32_t* status) {
  pdl_wait();
  pdl_trigger();
  const int64_t tok = blockIdx.x;
  const int D = c.head_dim, R = c.rope_dim, W = D + R;
  const int32_t slot = slots[tok];
  if (slot < 0) return;
  if ((int64_t)slot >= (int64_t)c.num_pages * c.page_size) {
    if (threadIdx.x == 0) set_status(status, KVQ_DEV_BAD_SLOT);
    return;
  }
  const int64_t r = (int64_t)(slot / c.page_size) * c.page_size + slot % c.page_size;
  __shared__ float red[2][4];
  float al = 0.f, ar = 0.f;
  for (int i = threadIdx.x; i < W; i += blockDim.x) {
    const float a = fabsf(load_act(rows, dtype, tok * W + i));
    if (i < D) al = fmaxf(al, a);
    else ar = fmaxf(ar, a);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    al = fmaxf(al, __shfl_xor_sync(0xffffffffu, al, o));
    ar = fmaxf(ar, __shfl_xor_sync(0xffffffffu, ar, o));
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) { red[0][w] = al; red[1][w] = ar; }
  __syncthreads();
  al = fmaxf(fmaxf(red[0][0], red[0][1]), fmaxf(red[0][2], red[0][3]));
  ar = fmaxf(fmaxf(red[1][0], red[1][1]), fmaxf(red[1][2], red[1][3]));
  const float invl = __fdiv_rn(448.0f, al), invr = __fdiv_rn(448.0f, ar);
  const bool zl = (al == 0.0f) || isinf(invl), zr = (ar == 0.0f) || isinf(invr);
  uint8_t* lc = static_cast<uint8_t*>(c.k) + r * D;
  uint8_t* rc = static_cast<uint8_t*>(c.v) + r * R;
  for (int i = threadIdx.x; i < W; i += blockDim.x) {
    const float x = load_act(rows, dtype, tok * W + i);
    if (i < D) lc[i] = zl ? 0 : e4m3_encode(__fmul_rn(x, invl));
    else rc[i - D] = zr ? 0 : e4m3_encode(__fmul_rn(x, invr));
  }
  if (threadIdx.x == 0) {
    static_cast<float*>(c.k_scale)[r] = __fdiv_rn(al, 448.0f);
    static_cast<float*>(c.v_scale)[r] = __fdiv_rn(ar, 448.0f);
  }
}

// y = blockdiag(H) x; one warp per 32-group (group g of the rows).
__device__ __forceinline__ void rotate_warp(const void* __restrict__ x, int dtype, float* y, int64_t n_groups,
                                            int64_t g) {
  const int lane = threadIdx.x & 31;
  if (g >= n_groups) return;
  float v = load_act(x, dtype, g * 32 + lane);
  v = warp_fwht32(v, lane);
  y[g * 32 + lane] = __fmul_rn(v, kHadamardScale);
}

__global__ void __launch_bounds__(256) rotate_kernel(const void* __restrict__ x, int dtype, float* y,
                                                     int64_t n_groups) {
  pdl_wait();
  pdl_trigger();
  rotate_warp(x, dtype, y, n_groups, (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5));
}

// The decode step's two independent preparations in one launch: blocks
// [0, store_blocks) run the store of the new tokens (one warp per (row,
// group)), the others rotate the queries.  Same arithmetic, same bytes as
// store_q4_group_kernel + rotate_kernel.
template <int NG>
__global__ void __launch_bounds__(256) store_rotate_kernel(kvq_cache c, const void* __restrict__ k,
                                                           const void* __restrict__ v, int dtype, int64_t n_tok,
                                                           const int32_t* __restrict__ slots, int32_t* status,
                                                           int store_blocks, const void* __restrict__ q,
                                                           int q_dtype, float* q_out, int64_t q_groups) {
  pdl_wait();
  pdl_trigger();
  const int warps = blockDim.x >> 5, w = threadIdx.x >> 5;
  if ((int)blockIdx.x < store_blocks)
    store_q4_group_warp<NG, true>(c, k, v, dtype, n_tok, slots, status, (int64_t)blockIdx.x * warps + w);
  else
    rotate_warp(q, q_dtype, q_out, q_groups, (int64_t)(blockIdx.x - store_blocks) * warps + w);
}

// ---------------------------------------------------------------- launchers

// Up to this many rows the store runs one warp per (row, group).
constexpr int64_t kStoreGroupRows = 256;

cudaError_t launch_store(const kvq_cache& c, const void* k, const void* v, int dtype, int64_t n_tok,
                         const int32_t* slots, int32_t* status, cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  const bool q4 = c.format == KVQ_FMT_Q4_HAD32 || c.format == KVQ_FMT_Q4_0;
  const bool rot = c.format == KVQ_FMT_Q4_HAD32;
  if (q4 && n_tok * c.num_kv_heads * 2 <= kStoreGroupRows) {
    const int64_t warps = n_tok * c.num_kv_heads * 2 * (c.head_dim / 32);
    const dim3 blocks((warps + 7) / 8);
#define KVQ_STORE_GROUP(NG)                                                                                      \
  e = rot ? launch_pdl(store_q4_group_kernel<NG, true>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status) \
          : launch_pdl(store_q4_group_kernel<NG, false>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status)
    switch (c.head_dim / 32) {
      case 1: KVQ_STORE_GROUP(1); break;
      case 2: KVQ_STORE_GROUP(2); break;
      case 4: KVQ_STORE_GROUP(4); break;
      case 8: KVQ_STORE_GROUP(8); break;
      default: return cudaErrorInvalidValue;
    }
#undef KVQ_STORE_GROUP
  } else if (q4) {
    const int64_t rows = n_tok * c.num_kv_heads * 2;
    const dim3 blocks((rows + 7) / 8);
#define KVQ_STORE_ROW(NG)                                                                                   \
  e = rot ? launch_pdl(store_q4_kernel<NG, true>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status) \
          : launch_pdl(store_q4_kernel<NG, false>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status)
    switch (c.head_dim / 32) {
      case 1: KVQ_STORE_ROW(1); break;
      case 2: KVQ_STORE_ROW(2); break;
      case 4: KVQ_STORE_ROW(4); break;
      case 8: KVQ_STORE_ROW(8); break;
      default: return cudaErrorInvalidValue;
    }
#undef KVQ_STORE_ROW
  } else if (c.format == KVQ_FMT_BF16) {
    const int64_t total = n_tok * c.num_kv_heads * c.head_dim;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 64) blocks = 152 * 64;
    e = launch_pdl(store_bf16_kernel, dim3(blocks), dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status);
  } else {
    e = launch_pdl(store_fp8_kernel, dim3(n_tok), dim3(128), 0, s, c, k, dtype, n_tok, slots, status);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool store_rotate_fits(const kvq_cache& c, int64_t n_tok) {
  const int ng = c.head_dim / 32;
  return c.format == KVQ_FMT_Q4_HAD32 && c.head_dim % 32 == 0 && n_tok * c.num_kv_heads * 2 <= kStoreGroupRows &&
         (ng == 1 || ng == 2 || ng == 4 || ng == 8);
}

cudaError_t launch_store_rotate(const kvq_cache& c, const void* k, const void* v, int dtype, int64_t n_tok,
                                const int32_t* slots, int32_t* status, const void* q, int q_dtype, float* q_out,
                                int64_t q_rows, int q_head_dim, cudaStream_t s) {
  const int64_t store_warps = n_tok * c.num_kv_heads * 2 * (c.head_dim / 32);
  const int store_blocks = static_cast<int>((store_warps + 7) / 8);
  const int64_t q_groups = q_rows * (q_head_dim / 32);
  const dim3 blocks(store_blocks + static_cast<unsigned>((q_groups + 7) / 8));
  if (blocks.x == 0) return cudaSuccess;
  cudaError_t e;
  switch (c.head_dim / 32) {
    case 1: e = launch_pdl(store_rotate_kernel<1>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status, store_blocks, q, q_dtype, q_out, q_groups); break;
    case 2: e = launch_pdl(store_rotate_kernel<2>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status, store_blocks, q, q_dtype, q_out, q_groups); break;
    case 4: e = launch_pdl(store_rotate_kernel<4>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status, store_blocks, q, q_dtype, q_out, q_groups); break;
    case 8: e = launch_pdl(store_rotate_kernel<8>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status, store_blocks, q, q_dtype, q_out, q_groups); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_rotate(const void* x, int dtype, float* y, int64_t rows, int head_dim, cudaStream_t s) {
  const int64_t groups = rows * (head_dim / 32);
  if (groups == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(rotate_kernel, dim3((groups + 7) / 8), dim3(256), 0, s, x, dtype, y, groups);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvq
