// tq4.cu -- the TQ4 rows: store (randomized Hadamard over the row, Lloyd-Max
// codebook at radius / sqrt(n)) and the signed row rotation of queries and
// outputs.
//
// Follows "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", PR body, "Why
// rotated-int4": a randomized-Hadamard rotation makes the coordinates of a row
// close to Gaussian and keeps its radius, so a fixed 16-level Lloyd-Max
// codebook for N(0,1), scaled by radius / sqrt(n), quantizes every coordinate
// with one scale per row.
//
// One warp per row; lane l holds elements E l .. E l + E - 1 (E = D / 32), so
// the butterfly's first log2(E) stages run in registers and the other five
// across lanes, and the pairwise tree of the sum of squares is the warp's
// xor reduction.  This TU is compiled with -fmad=false: the squares and sums
// round exactly as written.
#include "kernels.cuh"

namespace kvq {

namespace {

// Lloyd-Max magnitudes for 16 levels of N(0,1), rounded to fp16 (exact values).
__host__ __device__ constexpr float tq4_mag(int m) {
  return m == 0 ? 0.12841796875f : m == 1 ? 0.387939453125f : m == 2 ? 0.65673828125f : m == 3 ? 0.9423828125f
       : m == 4 ? 1.255859375f : m == 5 ? 1.6181640625f : m == 6 ? 2.068359375f : 2.732421875f;
}
// Midpoint between magnitudes m and m + 1 (exact: fp16 values summed in fp32).
__host__ __device__ constexpr float tq4_mid(int m) { return (tq4_mag(m) + tq4_mag(m + 1)) * 0.5f; }

template <int E>
__host__ __device__ constexpr float tq4_row_scale() {  // fp32(1 / sqrt(32 E))
  return E == 8 ? 0.0625f : E == 4 ? 0.0883883476483184405501f : 0.125f;
}

// In-place signed transform of the warp's row (forward: signs, butterfly, scale;
// inverse: butterfly, scale, signs).  `sw` holds this lane's E sign bits.
template <int E>
__device__ __forceinline__ void tq4_transform(float (&y)[E], uint32_t sw, int lane, bool inverse) {
  if (!inverse) {
#pragma unroll
    for (int i = 0; i < E; ++i)
      if ((sw >> i) & 1u) y[i] = -y[i];
  }
#pragma unroll
  for (int h = 1; h < E; h <<= 1)
#pragma unroll
    for (int i = 0; i < E; ++i)
      if (!(i & h)) {
        const float a = y[i], b = y[i + h];
        y[i] = __fadd_rn(a, b);
        y[i + h] = __fsub_rn(a, b);
      }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
#pragma unroll
    for (int i = 0; i < E; ++i) {
      const float p = __shfl_xor_sync(0xffffffffu, y[i], o);
      y[i] = (lane & o) ? __fsub_rn(p, y[i]) : __fadd_rn(y[i], p);
    }
#pragma unroll
  for (int i = 0; i < E; ++i) y[i] = __fmul_rn(y[i], tq4_row_scale<E>());
  if (inverse) {
#pragma unroll
    for (int i = 0; i < E; ++i)
      if ((sw >> i) & 1u) y[i] = -y[i];
  }
}

template <int E>
__device__ __forceinline__ uint32_t lane_signs(const void* signs, int lane) {
  const uint32_t w = static_cast<const uint32_t*>(signs)[(E * lane) >> 5];
  return w >> ((E * lane) & 31);
}

template <int E>
__global__ void __launch_bounds__(256) store_tq4_kernel(kvq_cache c, const void* __restrict__ k,
                                                        const void* __restrict__ v, int dtype, int64_t n_tok,
                                                        const int32_t* __restrict__ slots, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  constexpr int D = 32 * E;
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
  const int64_t r = ((int64_t)(slot / c.page_size) * Hk + head) * c.page_size + slot % c.page_size;
  const void* src = kv ? v : k;
  const int64_t base = (tok * Hk + head) * D + E * lane;

  float y[E];
#pragma unroll
  for (int i = 0; i < E; ++i) y[i] = load_act(src, dtype, base + i);
  tq4_transform<E>(y, lane_signs<E>(c.signs, lane), lane, false);

  // sum of squares by the pairwise tree: in-lane stages, then the xor reduction
  float q2[E];
#pragma unroll
  for (int i = 0; i < E; ++i) q2[i] = __fmul_rn(y[i], y[i]);
#pragma unroll
  for (int h = 1; h < E; h <<= 1)
#pragma unroll
    for (int i = 0; i < E; i += 2 * h) q2[i] = __fadd_rn(q2[i], q2[i + h]);
  float ss = q2[0];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, o));
  __half s16 = __float2half_rn(__fsqrt_rn(__fmul_rn(ss, 1.0f / D)));
  if (__hisinf(s16)) s16 = __ushort_as_half(0x7BFFu);  // saturate to 65504
  const float s = __half2float(s16);

  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    uint32_t code = 0;
    if (s > 0.0f) {
      const float q = __fdiv_rn(y[i], s);
      const float a = fabsf(q);
      uint32_t m = 0;
#pragma unroll
      for (int j = 0; j < 7; ++j) m += a > tq4_mid(j) ? 1u : 0u;
      code = (q < 0.0f ? 8u : 0u) | m;
    }
    word |= code << (4 * i);
  }
  uint8_t* codes = static_cast<uint8_t*>(kv ? c.v : c.k) + r * (D / 2) + lane * (E / 2);
  if constexpr (E == 8) {
    *reinterpret_cast<uint32_t*>(codes) = word;
  } else if constexpr (E == 4) {
    *reinterpret_cast<uint16_t*>(codes) = static_cast<uint16_t>(word);
  } else {
    *codes = static_cast<uint8_t>(word);
  }
  if (lane == 0) static_cast<__half*>(kv ? c.v_scale : c.k_scale)[r] = s16;
}

template <int E>
__global__ void __launch_bounds__(256) tq4_rotate_kernel(const void* __restrict__ signs, const void* x, int dtype,
                                                         float* y, int64_t rows, int inverse) {
  pdl_wait();
  pdl_trigger();
  constexpr int D = 32 * E;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= rows) return;
  float v[E];
#pragma unroll
  for (int i = 0; i < E; ++i) v[i] = load_act(x, dtype, row * D + E * lane + i);
  __syncwarp();  // every lane has read its inputs before any lane writes (y may alias x)
  tq4_transform<E>(v, lane_signs<E>(signs, lane), lane, inverse != 0);
#pragma unroll
  for (int i = 0; i < E; ++i) y[row * D + E * lane + i] = v[i];
}

}  // namespace

cudaError_t launch_store_tq4(const kvq_cache& c, const void* k, const void* v, int dtype, int64_t n_tok,
                             const int32_t* slots, int32_t* status, cudaStream_t s) {
  if (n_tok == 0) return cudaSuccess;
  const int64_t rows = n_tok * c.num_kv_heads * 2;
  const dim3 blocks(static_cast<unsigned>((rows + 7) / 8));
  cudaError_t e;
  switch (c.head_dim) {
    case 64: e = launch_pdl(store_tq4_kernel<2>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status); break;
    case 128: e = launch_pdl(store_tq4_kernel<4>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status); break;
    case 256: e = launch_pdl(store_tq4_kernel<8>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_tq4_rotate(const kvq_cache& c, const void* x, int dtype, float* y, int64_t rows, int inverse,
                              cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  const dim3 blocks(static_cast<unsigned>((rows + 7) / 8));
  cudaError_t e;
  switch (c.head_dim) {
    case 64: e = launch_pdl(tq4_rotate_kernel<2>, blocks, dim3(256), 0, s, c.signs, x, dtype, y, rows, inverse); break;
    case 128: e = launch_pdl(tq4_rotate_kernel<4>, blocks, dim3(256), 0, s, c.signs, x, dtype, y, rows, inverse); break;
    case 256: e = launch_pdl(tq4_rotate_kernel<8>, blocks, dim3(256), 0, s, c.signs, x, dtype, y, rows, inverse); break;
    default: return cudaErrorInvalidValue;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvq
