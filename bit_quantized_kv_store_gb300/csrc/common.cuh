// common.cuh -- device helpers shared by the libkvq kernels (sm_103a).
//
// Thin inline-PTX wrappers: mbarrier waits with an iteration bound, 1-D bulk
// (TMA) copies global -> shared, legacy warp-level MMA (m16n8k16 f16/bf16 ->
// f32), 8x8 b16 register transpose, and the status-word helpers.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <utility>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kPart = 512;  // keys per split-T partition ("shared 512-key chunks")
constexpr float kLog2e = 1.4426950408889634f;

// fp32 nearest value of 1/sqrt(32); the store multiplies by it once after the
// butterfly (0x3E3504F3).
constexpr float kHadamardScale = 0.17677669529663687f;

// ---------------------------------------------------------------- programmatic dependent launch
// Every kernel of the library calls pdl_wait() before it reads anything a
// kernel could have written and before any write: it returns once the
// preceding kernel in the stream has completed and its memory is visible (at
// once when there is none), so a kernel launched by launch_pdl may be
// scheduled while its predecessor drains without reading or overwriting
// anything early.  Only caller metadata that no kernel of the library writes
// (sequence lengths, block tables) may be read before it (the 4-bit decode
// does, to overlap those loads with the predecessor).  Every CTA calls it
// before it can exit, so the ordering is transitive along the stream.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the next kernel in the stream be scheduled now (its pdl_wait still waits
// for this whole grid to complete).  Small kernels call it at once; the large
// ones only near their end, so waiting successor CTAs never take their slots.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

__device__ __forceinline__ void set_status(int32_t* st, int32_t bit) {
  if (st) atomicOr(st, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (TMA) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Order this thread's generic-proxy global writes before later async-proxy
// (TMA, bulk copy) reads of them.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Add `bytes` to the current phase's expected transaction count, without an arrival.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// Asynchronous global -> shared copies through the load path (not the bulk-copy
// engine): 16 bytes cached in L2 only; 4 bytes, zero-filled past src_bytes.
// Both addresses aligned to the copy's size.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_4(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
// This thread's arrival on `bar`, made once every cp.async it issued before has
// landed (counts as one of the phase's expected arrivals).
__device__ __forceinline__ void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// The current phase of `bar` also waits for every cp.async this thread issued
// before (one more pending arrival now, made when they have landed; the phase's
// expected count is unchanged).  Must come before the phase can complete.
__device__ __forceinline__ void cp_async_mbar_track(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// 1-D bulk copy global -> shared, completing `bytes` transaction bytes on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar` to complete.  Gives up after ~2 s (the copies
// it waits for take microseconds) and returns false; the caller reports
// KVQ_DEV_TIMEOUT instead of hanging the GPU.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < (1u << 26); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && global_timer_ns() - t0 > 2000000000ull) break;
  }
  return false;
}

// ---------------------------------------------------------------- shared loads

__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(p)));
  return v;
}

// Element i of an activation tensor of dtype KVQ_DT_F32 or KVQ_DT_BF16, as fp32.
__device__ __forceinline__ float load_act(const void* p, int dtype, int64_t i) {
  if (dtype == KVQ_DT_F32) return static_cast<const float*>(p)[i];
  return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// ---------------------------------------------------------------- division by a launch constant
// n / d for 0 <= n < 2^31 and a divisor d >= 1 known at launch, as one
// multiply-high, an add and a shift (Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994: with l = ceil(log2 d)
// and m = floor(2^32 (2^l - d) / d) + 1, n / d = (mulhi(n, m) + n) >> l).
struct FastDiv {
  uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((uint64_t(1) << l) < d) ++l;
  const uint64_t m = ((uint64_t(1) << 32) * ((uint64_t(1) << l) - d)) / d + 1;
  return FastDiv{d, static_cast<uint32_t>(m), l};
}

__device__ __forceinline__ uint32_t fast_div(uint32_t n, const FastDiv& f) {
  return (__umulhi(n, f.m) + n) >> f.l;
}

// ---------------------------------------------------------------- register ops

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  return __byte_perm(a, b, sel);
}

// (a & b) | c  (lop3 with immLut 0xEA)
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// Two 4-bit codes (biased by 8) sitting in bits [0,4) and [16,20) of x -> the f16
// pair (c0 - 8, c1 - 8), exactly.  0x6400 | c is the f16 value 1024 + c.
__device__ __forceinline__ uint32_t nib_lo_pair(uint32_t x) {
  const uint32_t v = and_or(x, 0x000F000Fu, 0x64006400u);
  return h2_as_u32(__hsub2(u32_as_h2(v), u32_as_h2(0x64086408u)));  // - 1032
}
// Codes in bits [4,8) and [20,24): 0x6400 | (c << 4) is 1024 + 16c, so
// (1024 + 16c) / 16 - 72 = c - 8, exactly.
__device__ __forceinline__ uint32_t nib_hi_pair(uint32_t x) {
  const uint32_t v = and_or(x, 0x00F000F0u, 0x64006400u);
  return h2_as_u32(__hfma2(u32_as_h2(v), u32_as_h2(0x2C002C00u) /* 1/16 */, u32_as_h2(0xD480D480u) /* -72 */));
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  return h2_as_u32(__floats2half2_rn(lo, hi));
}

// Split x into an f16 high part and an f16 low part, x ~= hi + lo to ~22 bits.
__device__ __forceinline__ void split_f16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  hi = h2_as_u32(h);
  lo = pack_half2(x0 - hf.x, x1 - hf.y);
}

// ---------------------------------------------------------------- MMA

// D += A(16x16, row) * B(16x8, col); f16 inputs, f32 accumulate.  (Pure register
// operations are not `volatile`, so the compiler may interleave independent chains.)
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B + C with C given separately (the accumulator starts from C without
// a copy of C into D's registers; same arithmetic as mma_f16 on d = C).
__device__ __forceinline__ void mma_f16_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1, float c0, float c1, float c2, float c3) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%10,%11,%12,%13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose an 8x8 matrix of 16-bit values held one row-pair per thread.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

// 2^x with the hardware approximation (relative error ~2^-22; results below the
// smallest normal flush to zero, which only drops probabilities < 2^-126).
__device__ __forceinline__ float fast_exp2(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Two codes in bits [0,4) and [16,20) -> the f16 pair (1024 + c0, 1024 + c1), the
// 8 left in (the caller removes the bias elsewhere).
__device__ __forceinline__ uint32_t nib_lo_pair_biased(uint32_t x) { return and_or(x, 0x000F000Fu, 0x64006400u); }
// Codes in bits [4,8) and [20,24) -> (1024 + 16 c0, 1024 + 16 c1).
__device__ __forceinline__ uint32_t nib_hi_pair_biased(uint32_t x) { return and_or(x, 0x00F000F0u, 0x64006400u); }

// ---------------------------------------------------------------- warp FWHT

// In-register 32-point Walsh-Hadamard butterfly across a warp (lane i holds
// x[i]); stage order h = 1, 2, 4, 8, 16; lane i's new value is x[i] + x[i^h]
// when bit h of i is clear and x[i^h] - x[i] otherwise.  No scaling.
__device__ __forceinline__ float warp_fwht32(float x, int lane) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, x, h);
    x = (lane & h) ? __fsub_rn(o, x) : __fadd_rn(x, o);
  }
  return x;
}

}  // namespace kvq
