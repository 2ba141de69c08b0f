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
#include "q4_code.cuh"

namespace kvq {

// ---------------------------------------------------------------- packed fp32 pairs
// f32x2 instructions: two IEEE fp32 operations (round to nearest even), one per
// half, in one instruction -- the same results as the scalar forms.
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}

// One rotated group in registers: x[32] (the raw values) -> the 32 codes in
// word[0..3] (value 8q + i in nibble i of word q) and the fp16 scale; x ends as
// the rotated values y.  The butterfly runs on the pairs (x[i], x[i + 16]):
// stages 1, 2, 4, 8 pair registers i and i + h half by half, stage 16 adds the
// two halves of a register -- the same operations on the same operands as the
// scalar butterfly.  Codes: with t = fl(y * rcp(s) + 8) clamped to <= 15 (a t
// above 15 gives code 15 either way), u = fl(t + 1.5 * 2^23) holds rint_even(t)
// in its low mantissa bits (|t| < 2^22), and u - 1.5 * 2^23 - t is t's distance
// to it; the group takes these codes when every distance passes the screen
// (q4_code_screened's bound).  For an fp16-normal, unsaturated scale, t >= -1/2
// (|y| <= amax and s >= (amax / 8)(1 - 2^-11)), so no lower clamp is needed.
// Any other group (a distance near 1/2, a NaN or saturated or subnormal scale)
// takes the per-value screen and the IEEE division, as the other store forms do.
__device__ __forceinline__ void q4_group_rotated(float (&x)[32], uint32_t (&word)[4], __half& s16_out) {
  uint64_t P[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) P[i] = pk2(x[i], x[i + 16]);
#pragma unroll
  for (int h = 1; h < 16; h <<= 1)
#pragma unroll
    for (int i = 0; i < 16; ++i)
      if ((i & h) == 0) {
        const uint64_t a = P[i], b = P[i + h];
        P[i] = add2(a, b);
        P[i + h] = sub2(a, b);
      }
  const uint64_t C2 = pk2(kHadamardScale, kHadamardScale);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float a, b;
    upk2(P[i], a, b);
    P[i] = mul2(pk2(__fadd_rn(a, b), __fsub_rn(a, b)), C2);
    upk2(P[i], x[i], x[i + 16]);
  }
  // the group maximum by a tree (max is exact, so any order gives the same value)
  float m[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) m[i] = fmaxf(fabsf(x[i]), fabsf(x[i + 16]));
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  const float s32 = __fmul_rn(m[0], 0.125f);  // = amax / 8 correctly rounded (a power of two)
  __half s16 = __float2half_rn(s32);
  if (__hisinf(s16)) s16 = __ushort_as_half(0x7BFFu);  // saturate to 65504
  s16_out = s16;
  const float s = __half2float(s16);
  word[0] = word[1] = word[2] = word[3] = 0x88888888u;  // scale 0: every code 8
  if (s == 0.0f) return;
  const float r = rcp_approx(s);
  bool fast = s >= 6.103515625e-05f && s < 65504.0f;  // fp16-normal, unsaturated (false for NaN)
  if (fast) {
    const uint64_t R2 = pk2(r, r), E2 = pk2(8.0f, 8.0f), M2 = pk2(12582912.0f, 12582912.0f);
    float dmax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float ta, tb;
      upk2(fma2(P[i], R2, E2), ta, tb);
      const uint64_t t2 = pk2(fminf(ta, 15.0f), fminf(tb, 15.0f));
      const uint64_t u2 = add2(t2, M2);
      float da, db, ua, ub;
      upk2(sub2(t2, sub2(u2, M2)), da, db);
      dmax = fmaxf(dmax, fmaxf(fabsf(da), fabsf(db)));
      upk2(u2, ua, ub);
      word[i >> 3] = put_nibble(word[i >> 3], __float_as_uint(ua), i & 7);
      word[2 + (i >> 3)] = put_nibble(word[2 + (i >> 3)], __float_as_uint(ub), i & 7);
    }
    fast = dmax < kQ4Screen;
  }
  if (fast) return;
  word[0] = word[1] = word[2] = word[3] = 0x88888888u;
  uint32_t undecided = 0;  // bit i: value i needs the IEEE division
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t code;
      if (!q4_code_screened(x[8 * q + i], r, code)) undecided |= 1u << (8 * q + i);
      word[q] = put_nibble(word[q], code, i);
    }
  while (undecided) {
    const int i = __ffs(undecided) - 1;
    undecided &= undecided - 1;
    float y = x[0];
#pragma unroll
    for (int j = 1; j < 32; ++j)
      if (j == i) y = x[j];
    word[i >> 3] = put_nibble(word[i >> 3], q4_code_exact(y, s), i & 7);
  }
}

// Bulk form (a prompt chunk): one lane per (row, group of 32 values), so the
// whole 32-point butterfly (stages h = 1, 2, 4, 8, 16, (a, b) -> (a + b, a - b),
// the same operations on the same operands as the warp-shuffle form) and the
// group maximum run in registers, with no shuffles; consecutive lanes take
// consecutive groups.  The grid is sized to the GPU and every thread walks the
// groups with a grid stride, loading the next group's values before it
// quantises the current one, so the memory latency is paid once per thread and
// not once per group.  The lane's 16 code bytes and its fp16 scale are one
// 16-byte and one 2-byte store.  VEC: the inputs are 16-byte aligned (the
// lane loads its 32 values with 16-byte loads).  ROT = false: the unrotated
// Q4_0 format.  The launch keeps n_tok * num_kv_heads * 2 * NG below 2^31 (a
// larger store is split into several launches), so the group indices are
// 32-bit; hk and ps divide by num_kv_heads and page_size.
// The raw values of one group into w: 16 words of bf16 pairs (BF) or 32 f32.
template <bool VEC, bool BF>
__device__ __forceinline__ void load_group(const void* __restrict__ src, int dtype, int64_t e0,
                                           uint32_t (&w)[BF ? 16 : 32]) {
  if constexpr (BF) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 u = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + e0)[q];
      w[4 * q] = u.x; w[4 * q + 1] = u.y; w[4 * q + 2] = u.z; w[4 * q + 3] = u.w;
    }
  } else if constexpr (VEC) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 u = reinterpret_cast<const uint4*>(static_cast<const float*>(src) + e0)[q];
      w[4 * q] = u.x; w[4 * q + 1] = u.y; w[4 * q + 2] = u.z; w[4 * q + 3] = u.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(load_act(src, dtype, e0 + i));
  }
}

// BF: bf16 inputs with VEC (16-byte loads of bf16 pairs); otherwise 32 f32 words
// (VEC) or element loads of either type.
constexpr int kLaneBlock = 128;

template <int NG, bool ROT, bool VEC, bool BF = false>
__global__ void __launch_bounds__(kLaneBlock, 5) store_q4_lane_kernel(kvq_cache c, const void* __restrict__ k,
                                                            const void* __restrict__ v, int dtype, int64_t n_tok,
                                                            const int32_t* __restrict__ slots, int32_t* status,
                                                            FastDiv hk, FastDiv ps) {
  pdl_wait();
  pdl_trigger();
  constexpr int D = NG * 32;
  const int Hk = c.num_kv_heads;
  const uint32_t total = static_cast<uint32_t>(n_tok * Hk * 2 * NG);
  const uint32_t stride = gridDim.x * blockDim.x;
  // where group gg's values start, and which plane it goes to
  auto locate = [&](uint32_t gg, uint32_t& tok, uint32_t& head, bool& is_v) -> int64_t {
    const uint32_t row = gg / NG, rowh = row >> 1;
    tok = fast_div(rowh, hk);
    head = rowh - tok * Hk;
    is_v = (row & 1) != 0;
    return ((int64_t)tok * Hk + head) * D + 32 * static_cast<int>(gg % NG);
  };
  uint32_t gg = blockIdx.x * blockDim.x + threadIdx.x;
  uint32_t nxt[BF ? 16 : 32];  // the next group's raw values
  int32_t nslot = -1;          // and its token's slot
  if (gg < total) {
    uint32_t tok, head;
    bool is_v;
    const int64_t e0 = locate(gg, tok, head, is_v);
    load_group<VEC, BF>(is_v ? v : k, dtype, e0, nxt);
    nslot = slots[tok];
  }
  for (; gg < total; gg += stride) {
    uint32_t tok, head;
    bool is_v;
    locate(gg, tok, head, is_v);
    const int G = static_cast<int>(gg % NG);
    const int32_t slot = nslot;
    float x[32];
    if constexpr (BF) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        x[2 * i] = __uint_as_float(nxt[i] << 16);
        x[2 * i + 1] = __uint_as_float(nxt[i] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(nxt[i]);
    }
    if (gg + stride < total) {  // the next group's loads go ahead of this group's arithmetic
      uint32_t t2, h2;
      bool v2;
      const int64_t e2 = locate(gg + stride, t2, h2, v2);
      load_group<VEC, BF>(v2 ? v : k, dtype, e2, nxt);
      nslot = slots[t2];
    }
    // the codes first: only the stores depend on the slot
    uint32_t word[4];
    __half s16;
    if constexpr (ROT) {
      q4_group_rotated(x, word, s16);
    } else {
    // the group maximum by a tree (max is exact, so any order gives the same value)
    float m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = fmaxf(fabsf(x[i]), fabsf(x[i + 16]));
#pragma unroll
    for (int w = 8; w > 0; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
    const float amax = m[0];
    const float s32 = __fmul_rn(amax, 0.125f);  // = amax / 8 correctly rounded (a power of two)
    s16 = __float2half_rn(s32);
    if (__hisinf(s16)) s16 = __ushort_as_half(0x7BFFu);  // saturate to 65504
    const float s = __half2float(s16);
    word[0] = word[1] = word[2] = word[3] = 0x88888888u;  // scale 0: every code 8
    if (s != 0.0f) {
      const float r = rcp_approx(s);
      uint32_t undecided = 0;  // bit i: value i needs the IEEE division
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint32_t code;
          if (!q4_code_screened(x[8 * q + i], r, code)) undecided |= 1u << (8 * q + i);
          word[q] = put_nibble(word[q], code, i);
        }
      }
      // ties and near-ties (rare after the rotation; frequent for unrotated
      // inputs of few mantissa bits, where y / s is often exactly k + 1/2):
      // only those values take the division
      while (undecided) {
        const int i = __ffs(undecided) - 1;
        undecided &= undecided - 1;
        float y = x[0];
#pragma unroll
        for (int j = 1; j < 32; ++j)
          if (j == i) y = x[j];
        word[i >> 3] = put_nibble(word[i >> 3], q4_code_exact(y, s), i & 7);
      }
    }
    }
    if (slot < 0) continue;
    if ((int64_t)slot >= (int64_t)c.num_pages * c.page_size) {
      if (G == 0) set_status(status, KVQ_DEV_BAD_SLOT);
      continue;
    }
    const uint32_t page = fast_div(static_cast<uint32_t>(slot), ps);
    const int64_t r = ((int64_t)page * Hk + head) * c.page_size + (static_cast<uint32_t>(slot) - page * ps.d);
    reinterpret_cast<uint4*>(static_cast<uint8_t*>(is_v ? c.v : c.k) + r * (D / 2))[G] =
        make_uint4(word[0], word[1], word[2], word[3]);
    (static_cast<uint16_t*>(is_v ? c.v_scale : c.k_scale) + r * NG)[G] = __half_as_ushort(s16);
  }
}

// Latency form of the same store for a handful of rows (a decode step stores one
// token): one warp per (row, group), so the groups of a row are packed in
// parallel instead of one after another.  Same arithmetic, same bytes.
// Warp `wid` of the store: (row, group) = (wid / NG, wid % NG).
// (n_tok * num_kv_heads * 2 * NG is at most a few thousand here; hk and ps
// divide by num_kv_heads and page_size.)
template <int NG, bool ROT>
__device__ __forceinline__ void store_q4_group_warp(const kvq_cache& c, const void* __restrict__ k,
                                                    const void* __restrict__ v, int dtype, int64_t n_tok,
                                                    const int32_t* __restrict__ slots, int32_t* status, int64_t wid,
                                                    const FastDiv& hk, const FastDiv& ps) {
  constexpr int D = NG * 32;
  const int lane = threadIdx.x & 31;
  const int Hk = c.num_kv_heads;
  if (wid >= n_tok * Hk * 2 * NG) return;
  const int G = static_cast<int>(wid % NG);
  const uint32_t row = static_cast<uint32_t>(wid / NG), rowh = row >> 1;
  const int kv = static_cast<int>(row & 1);
  const uint32_t tok = fast_div(rowh, hk);
  const int head = static_cast<int>(rowh - tok * Hk);
  const int32_t slot = slots[tok];
  if (slot < 0) return;
  if ((int64_t)slot >= (int64_t)c.num_pages * c.page_size) {
    if (lane == 0 && G == 0) set_status(status, KVQ_DEV_BAD_SLOT);
    return;
  }
  const uint32_t page = fast_div(static_cast<uint32_t>(slot), ps);
  const int off = static_cast<int>(static_cast<uint32_t>(slot) - page * ps.d);
  const int64_t r = ((int64_t)page * Hk + head) * c.page_size + off;
  const void* src = kv ? v : k;
  const float x = load_act(src, dtype, ((int64_t)tok * Hk + head) * D + 32 * G + lane);
  __half s16;
  const uint32_t code = q4_group_code_warp<ROT>(x, lane, s16);
  q4_write_group_warp(static_cast<uint8_t*>(kv ? c.v : c.k) + r * (D / 2),
                      static_cast<uint16_t*>(kv ? c.v_scale : c.k_scale) + r * NG, G, code, s16, lane);
}

template <int NG, bool ROT>
__global__ void __launch_bounds__(256) store_q4_group_kernel(kvq_cache c, const void* __restrict__ k,
                                                             const void* __restrict__ v, int dtype, int64_t n_tok,
                                                             const int32_t* __restrict__ slots, int32_t* status,
                                                             FastDiv hk, FastDiv ps) {
  pdl_wait();
  pdl_trigger();
  store_q4_group_warp<NG, ROT>(c, k, v, dtype, n_tok, slots, status,
                               (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), hk, ps);
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
                                                           int q_dtype, float* q_out, int64_t q_groups, FastDiv hk,
                                                           FastDiv ps) {
  pdl_wait();
  pdl_trigger();
  const int warps = blockDim.x >> 5, w = threadIdx.x >> 5;
  if ((int)blockIdx.x < store_blocks)
    store_q4_group_warp<NG, true>(c, k, v, dtype, n_tok, slots, status, (int64_t)blockIdx.x * warps + w, hk, ps);
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
  const FastDiv hk = make_fastdiv(static_cast<uint32_t>(c.num_kv_heads));
  const FastDiv ps = make_fastdiv(static_cast<uint32_t>(c.page_size));
  if (q4 && n_tok * c.num_kv_heads * 2 <= kStoreGroupRows) {
    const int64_t warps = n_tok * c.num_kv_heads * 2 * (c.head_dim / 32);
    const dim3 blocks((warps + 7) / 8);
#define KVQ_STORE_GROUP(NG)                                                                                        \
  e = rot ? launch_pdl(store_q4_group_kernel<NG, true>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status, \
                       hk, ps)                                                                                       \
          : launch_pdl(store_q4_group_kernel<NG, false>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots,      \
                       status, hk, ps)
    switch (c.head_dim / 32) {
      case 1: KVQ_STORE_GROUP(1); break;
      case 2: KVQ_STORE_GROUP(2); break;
      case 4: KVQ_STORE_GROUP(4); break;
      case 8: KVQ_STORE_GROUP(8); break;
      default: return cudaErrorInvalidValue;
    }
#undef KVQ_STORE_GROUP
  } else if (q4) {
    // one lane per (row, group); launches of at most 2^30 groups, so that the
    // kernel's group indices stay 32-bit
    int n_sm = device_sm_count(), per_sm = 0;
    if (n_sm < 1) n_sm = 1;
    {
      auto kern = rot ? store_q4_lane_kernel<8, true, true, true> : store_q4_lane_kernel<8, false, true, true>;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kLaneBlock, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    }
    const int64_t lane_threads = static_cast<int64_t>(n_sm) * per_sm * kLaneBlock;  // resident at once
    const int64_t per_tok = static_cast<int64_t>(c.num_kv_heads) * 2 * (c.head_dim / 32);
    const int64_t max_tok = (int64_t(1) << 30) / per_tok;
    const size_t esz = dtype == KVQ_DT_F32 ? 4 : 2;
    const size_t tok_bytes = static_cast<size_t>(c.num_kv_heads) * c.head_dim * esz;
    const bool vec = (reinterpret_cast<uintptr_t>(k) & 15u) == 0 && (reinterpret_cast<uintptr_t>(v) & 15u) == 0 &&
                     tok_bytes % 16 == 0;
    for (int64_t t0 = 0; t0 < n_tok && e == cudaSuccess; t0 += max_tok) {
      const int64_t nt = n_tok - t0 < max_tok ? n_tok - t0 : max_tok;
      const void* kc = static_cast<const uint8_t*>(k) + t0 * tok_bytes;
      const void* vc = static_cast<const uint8_t*>(v) + t0 * tok_bytes;
      const int32_t* sc = slots + t0;
      // a grid the GPU holds at once, every thread walking the same number of groups
      const int64_t groups = nt * per_tok;
      const int64_t per_thread = (groups + lane_threads - 1) / lane_threads;
      const dim3 blocks(static_cast<unsigned>((groups + per_thread * kLaneBlock - 1) / (per_thread * kLaneBlock)));
#define KVQ_STORE_WIDE(NG, ROT)                                                                                      \
  e = !vec ? launch_pdl(store_q4_lane_kernel<NG, ROT, false>, blocks, dim3(kLaneBlock), 0, s, c, kc, vc, dtype, nt, sc,     \
                        status, hk, ps)                                                                              \
    : dtype == KVQ_DT_BF16                                                                                           \
        ? launch_pdl(store_q4_lane_kernel<NG, ROT, true, true>, blocks, dim3(kLaneBlock), 0, s, c, kc, vc, dtype, nt, sc,   \
                     status, hk, ps)                                                                                 \
        : launch_pdl(store_q4_lane_kernel<NG, ROT, true, false>, blocks, dim3(kLaneBlock), 0, s, c, kc, vc, dtype, nt, sc,  \
                     status, hk, ps)
#define KVQ_STORE_ROW(NG)         \
  if (rot) {                      \
    KVQ_STORE_WIDE(NG, true);     \
  } else {                        \
    KVQ_STORE_WIDE(NG, false);    \
  }
      switch (c.head_dim / 32) {
        case 1: KVQ_STORE_ROW(1); break;
        case 2: KVQ_STORE_ROW(2); break;
        case 4: KVQ_STORE_ROW(4); break;
        case 8: KVQ_STORE_ROW(8); break;
        default: return cudaErrorInvalidValue;
      }
#undef KVQ_STORE_ROW
#undef KVQ_STORE_WIDE
    }
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
  const FastDiv hk = make_fastdiv(static_cast<uint32_t>(c.num_kv_heads));
  const FastDiv ps = make_fastdiv(static_cast<uint32_t>(c.page_size));
  cudaError_t e;
  switch (c.head_dim / 32) {
    case 1: e = launch_pdl(store_rotate_kernel<1>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status, store_blocks, q, q_dtype, q_out, q_groups, hk, ps); break;
    case 2: e = launch_pdl(store_rotate_kernel<2>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status, store_blocks, q, q_dtype, q_out, q_groups, hk, ps); break;
    case 4: e = launch_pdl(store_rotate_kernel<4>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status, store_blocks, q, q_dtype, q_out, q_groups, hk, ps); break;
    case 8: e = launch_pdl(store_rotate_kernel<8>, blocks, dim3(256), 0, s, c, k, v, dtype, n_tok, slots, status, store_blocks, q, q_dtype, q_out, q_groups, hk, ps); break;
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
