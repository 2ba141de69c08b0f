// q4_code.cuh -- the 4-bit code of a value and the quantization of one
// 32-value group across a warp, shared by the store kernels and the decode
// kernels that store a new token themselves.  Every floating-point operation
// here is an explicit IEEE-rounded intrinsic (no contraction), so the codes are
// the same bits whatever the including translation unit's -fmad setting.
#pragma once
#include "common.cuh"

namespace kvq {

// ---------------------------------------------------------------- the 4-bit code of one value
// code = clamp(rint_even(fl(y / s)), -8, 7) + 8, with fl(y / s) the IEEE-rounded
// fp32 quotient and s > 0 (an fp16 value, so a normal fp32 number).
//
// Screen: with r = rcp.approx(s) (at most 1 ulp off, PTX ISA), t = fl(y * r + 8)
// (one fused rounding) is within |Q| 2^-23 + |Q + 8| 2^-24 < 2^-18 of Q + 8
// while |Q| < 16, Q = y / s exactly, and fl(Q) is within 2^-21 of Q.  So when
// t is farther than 2^-14 from every half-integer, Q + 8 and fl(Q) + 8 lie
// strictly inside the same unit interval (k - 1/2, k + 1/2) around k = rint(t),
// and rint_even(fl(Q)) = k - 8 without a tie (8 is even, so ties keep their
// side).  For Q >= 16 (Q <= -16) both k and rint(fl(Q)) + 8 are beyond the
// clamp at 15 (at 0).  Anything else -- exact or near ties, NaN, infinities --
// takes the IEEE division.
constexpr float kQ4Screen = 0.5f - 0.00006103515625f;  // 1/2 - 2^-14

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// The code from the screened estimate; returns false when the estimate cannot
// decide it (then call q4_code_exact).
__device__ __forceinline__ bool q4_code_screened(float y, float r, uint32_t& code) {
  const float t = __fmaf_rn(y, r, 8.0f);
  const float k = rintf(t);
  code = static_cast<uint32_t>(fminf(fmaxf(k, 0.0f), 15.0f));
  return fabsf(__fsub_rn(t, k)) < kQ4Screen;
}

// Insert a 4-bit code at bit 4i of w.
__device__ __forceinline__ uint32_t put_nibble(uint32_t w, uint32_t code, int i) {
  uint32_t r;
  asm("bfi.b32 %0, %1, %2, %3, 4;" : "=r"(r) : "r"(code), "r"(w), "r"(4 * i));
  return r;
}

__device__ __forceinline__ uint32_t q4_code_exact(float y, float s) {
  float q = rintf(__fdiv_rn(y, s));
  q = fminf(fmaxf(q, -8.0f), 7.0f);
  return static_cast<uint32_t>(static_cast<int>(q) + 8);
}

// One 32-value group across a warp (lane i holds value i of the raw row): the
// group rotated (ROT) by the butterfly and the multiply by fp32(1/sqrt(32)),
// its fp16 scale fp16_rne(amax / 8) saturated to 65504 (into s16), and this
// lane's 4-bit code (8 everywhere for a zero scale).
template <bool ROT>
__device__ __forceinline__ uint32_t q4_group_code_warp(float x, int lane, __half& s16) {
  const float y = ROT ? __fmul_rn(warp_fwht32(x, lane), kHadamardScale) : x;
  float amax = fabsf(y);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s32 = __fmul_rn(amax, 0.125f);  // = amax / 8 correctly rounded (a power of two)
  s16 = __float2half_rn(s32);
  if (__hisinf(s16)) s16 = __ushort_as_half(0x7BFFu);  // saturate to 65504
  const float s = __half2float(s16);
  uint32_t code = 8;
  if (s != 0.0f && !q4_code_screened(y, rcp_approx(s), code)) code = q4_code_exact(y, s);
  return code;
}

// Write group G of a row: the 32 lanes' codes as the group's 16 bytes at
// codes_row + 16 G (value 2b in the low nibble of byte b) and the scale at
// scales_row[G].
__device__ __forceinline__ void q4_write_group_warp(uint8_t* codes_row, uint16_t* scales_row, int G, uint32_t code,
                                                    __half s16, int lane) {
  uint32_t bits = code << (4 * (lane & 3));
  bits |= __shfl_xor_sync(0xffffffffu, bits, 1);
  bits |= __shfl_xor_sync(0xffffffffu, bits, 2);
  if ((lane & 3) == 0) {
    const int h = lane >> 2;  // half-word h of group G: bytes 16G + 2h, 16G + 2h + 1
    reinterpret_cast<uint16_t*>(codes_row)[8 * G + h] = static_cast<uint16_t>(bits);
  }
  if (lane == 0) scales_row[G] = __half_as_ushort(s16);
}

}  // namespace kvq
