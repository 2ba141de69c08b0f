// decode_q4.cu -- split-T decode attention over the 4-bit caches.
//
// Follows "qwen27 CUDA: an opt-in 4-bit attention cache (262K on a 24 GB card)",
// section "What it is": attend over the 4-bit cache in rotated space, in shared
// 512-key chunks plus the tail, producing per-chunk partials that are merged in
// order; and "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", split-T
// commit: (H, P) partial online-softmax blocks (cl, m, z) + a log-sum-exp merge
// (and, for the TQ4 rows, its "Why rotated-int4" codebook).
//
// GB300 design.  One CTA of 4 warps per (partition of 512 keys, KV head,
// sequence), 4 CTAs per SM (128 registers, 48 KB of shared memory); a grid that
// fits in one wave of two CTAs per SM (a short context) runs a warp-specialised
// form instead (below: 4 scoring and 4 P.V warps per CTA, same arithmetic).  The
// partition is walked in rounds of 8 tiles of 16 keys (128 keys):
//  * Fragments: a code row is 8 groups of 16 bytes, so the 8 rows x 16 bytes of
//    an ldmatrix 8x8 matrix are one group of 8 keys: one ldmatrix.x4 gives a
//    thread its K words of two groups for keys g and g + 8, one
//    ldmatrix.x4.trans its V words for keys 2t, 2t+1, 2t+8, 2t+9.
//  * Scores: warp w takes tiles 2w, 2w + 1 of the round, all 256 dims, on the
//    tensor cores (mma.m16n8k16, the 16 keys of a tile on M, the <= 8 query
//    heads of the GQA group on N).  The key codes enter as the exact f16
//    values 1024 + c / 1024 + 16c (one lop3 per pair, the pairs taken from the
//    word by masks and one byte shift); the constant part is removed by
//    starting each group's accumulator at a per-(head, group) query bias.  The
//    query is split into f16 high and low parts (~22 bits; its fragments sit
//    in shared memory and are loaded once for both tiles); each 32-value
//    group gets its own partial product multiplied by the group's fp32 scale,
//    so the dequantised keys enter exactly.
//  * The warps exchange their maxima through shared memory, so that every warp
//    holds the same running maximum (base 2; the query carries
//    sm_scale * log2 e), and publish their probabilities as ready-made B
//    fragments (transposed in registers by movmatrix).
//  * Context: warp w owns value dims [64w, 64w + 64) (groups 2w, 2w + 1) and
//    runs P.V over all 8 tiles of the round, value dims on M: the
//    probabilities are multiplied by the V group scale in f16; V codes minus 8
//    are exact in f16.  Each thread keeps 16 accumulators; a rescale costs 18
//    FMULs.  Two named barriers per round.
//  * The sums of the probabilities are kept per tile slot (tile u of every
//    round) and added slot by slot at the end, in the same order in both forms.
// Modes of the same kernel: the gather of selected rows (GATHER); decode
// windows (WIN: up to 4 column tiles of (row, head) pairs of several rows of
// one sequence per CTA, each row masked at its own end); TQ4 rows (TQ: the
// nibbles become fp16 codebook levels by prmt lookups, one scale per row, V
// transposed per key pair by movmatrix).
// Copies: a tile of codes (16 rows x 128 B) arrives by a 2-D TMA tensor copy
// with the hardware 128-byte swizzle (16-byte chunk c of row r lands at chunk
// c ^ (r & 7), so the fragment loads are free of bank conflicts), its scales
// by a 1-D bulk copy; the gather variant copies row by row with 1-D bulk
// copies into rows padded to 144 bytes.  The rings hold one round: a warp
// refills its own K tiles right after its scores, and its share of the V tiles
// once an mbarrier shows every warp done with the round's P.V (a round takes
// microseconds, so the copies have ample lead).
#include <type_traits>

#include "kernels.cuh"
#include "q4_code.cuh"

namespace kvq {

constexpr int kQ4D = 256;
constexpr int kQ4NG = 8;
constexpr int kQ4TileBytes = 16 * 128;  // codes of one 16-key tile (dense: TMA, 128-byte swizzle)
constexpr int kQ4GatherRow = 144;       // gather: rows padded to 144 bytes (no swizzle), so that the
                                        // 8 rows of an ldmatrix fall in 8 distinct bank quads
// Bytes of one code tile in shared memory
template <bool GATHER>
__host__ __device__ constexpr int q4_tile_bytes() { return GATHER ? 16 * kQ4GatherRow : kQ4TileBytes; }
constexpr int kQ4ScaleBytes = 16 * 16;  // fp16 scales of one 16-key tile
constexpr float kQ4NoMax = -1e30f;      // softmax reference before the first key (finite: no -inf - -inf)

__device__ __forceinline__ void tma_rows_2d(void* dst, const CUtensorMap* map, int row, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(smem_u32(bar))
      : "memory");
}


// shared-memory loads at a 32-bit shared address
__device__ __forceinline__ uint4 lds128a(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t lds32a(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 lds64a(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ float2 lds64f(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}

// Four 8x8 matrices of 16-bit elements; lane l gives the address of row l & 7 of
// matrix l >> 3 (16 contiguous bytes).  Plain: lane (g, t) receives elements
// (g, 2t), (g, 2t + 1) of each matrix.  Transposed: elements (2t, g), (2t + 1, g).
__device__ __forceinline__ uint4 ldsm_x4(uint32_t addr) {
  uint4 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 ldsm_x4_trans(uint32_t addr) {
  uint4 v;
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// The fragments from this lane's query values u0 = q[8t .. 8t+3], u1 =
// q[8t+4 .. 8t+7] of each group G = warp + kWarps k (k < 8 / kWarps) of its
// column's query row (live = false: a dead column, zero query).
template <int kWarps>
__device__ __forceinline__ void q4_frag_build(const float4* ql0, const float4* ql1, bool live, float qscale,
                                              int warp, int lane, uint4 (*qf)[2][32], float4 (*qb)[4]) {
  const int g = lane >> 2, t = lane & 3;
  // The K codes enter the MMA as 1024 + c (even elements, low nibbles) and
  // 1024 + 16c (odd elements, high nibbles), one lop3 each; the query values
  // facing high nibbles are pre-divided by 16 (exact), and the accumulator of
  // group G starts at -bias_G, bias_G = 1024 * sum(B) + 8 * sum(q~) over the
  // group (B the f16 values in the fragments, q~ = B or 16 B), so the MMA
  // returns sum_d q_d (c_d - 8) with the keys' codes used exactly.
  const float s = live ? qscale : 0.f;
  const float s16 = s * 0.0625f;
  constexpr int kGroupsPerWarp = kQ4NG / kWarps;
#pragma unroll
  for (int k = 0; k < kGroupsPerWarp; ++k) {
    const int G = warp + kWarps * k;
    const float4 u0 = ql0[k];
    const float4 u1 = ql1[k];
    uint4 hi, lo;
    // first MMA of the group: slots (2t, 2t+1) <- d (8t, 8t+4) (low nibbles of
    // bytes 0, 2 of the key's word), slots (2t+8, 2t+9) <- d (8t+1, 8t+5) (high
    // nibbles); second MMA: d + 2 (the word shifted by a byte)
    split_f16(u0.x * s, u1.x * s, hi.x, lo.x);
    split_f16(u0.y * s16, u1.y * s16, hi.y, lo.y);
    split_f16(u0.z * s, u1.z * s, hi.z, lo.z);
    split_f16(u0.w * s16, u1.w * s16, hi.w, lo.w);
    qf[G][0][lane] = hi;
    qf[G][1][lane] = lo;
    float ev = 0.f, od = 0.f;  // sums of the even-slot and odd-slot B values (hi parts, then lo parts)
    const uint32_t hv[4] = {hi.x, hi.y, hi.z, hi.w}, lv[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float2 h2 = __half22float2(u32_as_h2(hv[r]));
      if (r & 1) od += h2.x + h2.y; else ev += h2.x + h2.y;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float2 l2 = __half22float2(u32_as_h2(lv[r]));
      if (r & 1) od += l2.x + l2.y; else ev += l2.x + l2.y;
    }
    // bias = 1024 (ev + od) + 8 (ev + 16 od), summed over the 4 lanes of the column
    float bias = 1032.f * ev + 1152.f * od;
    bias += __shfl_xor_sync(0xffffffffu, bias, 1);
    bias += __shfl_xor_sync(0xffffffffu, bias, 2);
    // column g's bias -> components (g & 1) and 2 + (g & 1) of qb[G][g / 2]
    if (t == 0) {
      float* q4 = reinterpret_cast<float*>(&qb[G][g >> 1]);
      q4[g & 1] = -bias;
      q4[2 + (g & 1)] = -bias;
    }
  }
}

// Query fragments (B operand of the score MMA) and biases of one column tile:
// column g of the tile faces the query row `qrow` (all 256 dims; a dead column
// passes live = false and gets a zero query).  Warp w prepares groups w,
// w + kWarps, ...; the caller synchronises before the fragments are read.
template <int kWarps>
__device__ __forceinline__ void q4_frag_prep(const float* qrow, bool live, float qscale, int warp, int lane,
                                             uint4 (*qf)[2][32], float4 (*qb)[4]) {
  const int t = lane & 3;
  constexpr int kGroupsPerWarp = kQ4NG / kWarps;
  float4 ql0[kGroupsPerWarp], ql1[kGroupsPerWarp];  // all loads issued first
#pragma unroll
  for (int k = 0; k < kGroupsPerWarp; ++k) {
    ql0[k] = *reinterpret_cast<const float4*>(qrow + 32 * (warp + kWarps * k) + 8 * t);
    ql1[k] = *reinterpret_cast<const float4*>(qrow + 32 * (warp + kWarps * k) + 8 * t + 4);
  }
  q4_frag_build<kWarps>(ql0, ql1, live, qscale, warp, lane, qf, qb);
}

// The round kernel's query preparation: an unrotated query is rotated one
// (head, group) pair per warp, lane = element, through a shared-memory scratch
// (qrot) and then built into fragments.  (The warp-specialised kernel rotates in
// the fragments' layout instead, below; in the round kernel that form measured
// 0.7 us slower at 262K keys, though its rotated-query path is the same.)
template <int kWarps>
struct RoundQueryLoads {
  float xs[8 * kQ4NG / kWarps];     // unrotated queries: the lane's element of each (head, group) pair
  float4 u0[kQ4NG / kWarps], u1[kQ4NG / kWarps];  // rotated queries: the lane's fragment inputs
};

template <int kWarps>
__device__ __forceinline__ void q4r_query_load(const DecodeArgs& a, int b, int kvh, int warp, int lane,
                                              RoundQueryLoads<kWarps>& L) {
  if (a.q_raw) {
    // warp w takes (head, group) pairs w, w + kWarps, ..., lane = element
    constexpr int kPairs = 8 * kQ4NG / kWarps;
    const int npairs = a.group * kQ4NG;
    const int64_t qbase = ((int64_t)b * a.Hq + kvh * a.group) * kQ4D + lane;
#pragma unroll
    for (int k = 0; k < kPairs; ++k) {
      const int hg = warp + kWarps * k;  // (head, group) = (hg / 8, hg % 8): elements 32 hg .. of the rows
      L.xs[k] = 0.f;
      if (hg < npairs)
        L.xs[k] = a.q_dtype == KVQ_DT_F32
                      ? static_cast<const float*>(a.q_raw)[qbase + 32 * hg]
                      : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q_raw)[qbase + 32 * hg]);
    }
  } else {
    const int g = lane >> 2, t = lane & 3;
    const float* qrow = a.q + ((int64_t)b * a.Hq + kvh * a.group + (g < a.group ? g : 0)) * kQ4D;
#pragma unroll
    for (int k = 0; k < kQ4NG / kWarps; ++k) {
      L.u0[k] = *reinterpret_cast<const float4*>(qrow + 32 * (warp + kWarps * k) + 8 * t);
      L.u1[k] = *reinterpret_cast<const float4*>(qrow + 32 * (warp + kWarps * k) + 8 * t + 4);
    }
  }
}

template <int kWarps>
__device__ __forceinline__ void q4r_query_build(const DecodeArgs& a, int warp, int lane, const RoundQueryLoads<kWarps>& L,
                                               float* qrot, uint4 (*qf)[2][32], float4 (*qb)[4]) {
  const int g = lane >> 2;
  const bool live = g < a.group;
  if (a.q_raw) {
    // Rotate with the arithmetic of the rotation entry point (fp32 butterfly,
    // stages 1..16, one multiply by fp32(1/sqrt(32))), through qrot (8 heads x
    // 256 fp32 of shared memory), then build the fragments from it.
    constexpr int kPairs = 8 * kQ4NG / kWarps;
    const int npairs = a.group * kQ4NG;
#pragma unroll
    for (int k = 0; k < kPairs; ++k) {
      const int hg = warp + kWarps * k;
      if (hg < npairs)  // warp-uniform
        qrot[32 * hg + lane] = a.q_rotate ? __fmul_rn(warp_fwht32(L.xs[k], lane), kHadamardScale) : L.xs[k];
    }
    __syncthreads();
    q4_frag_prep<kWarps>(qrot + (live ? g : 0) * kQ4D, live, a.qscale, warp, lane, qf, qb);
  } else {
    q4_frag_build<kWarps>(L.u0, L.u1, live, a.qscale, warp, lane, qf, qb);
  }
  __syncthreads();
}

// Both halves at once (the round kernel).
template <int kWarps>
__device__ __forceinline__ void q4r_query_prep(const DecodeArgs& a, int b, int kvh, int warp, int lane, float* qrot,
                                              uint4 (*qf)[2][32], float4 (*qb)[4]) {
  RoundQueryLoads<kWarps> L;
  q4r_query_load<kWarps>(a, b, kvh, warp, lane, L);
  q4r_query_build<kWarps>(a, warp, lane, L, qrot, qf, qb);
}

// The query preparation of one sequence's GQA group (columns = its heads) in two
// halves, so that a kernel can issue the global loads early and build the
// fragments later: q4_query_load issues them (into registers, not waited for);
// q4_query_build rotates the group's queries when they come unrotated and writes
// the fragments into qf / qb, ending with __syncthreads.  Thread (g, t) of warp
// w holds, for head g and each of its groups G = w, w + kWarps, ..., the 8
// values 32 G + 8 t .. + 7: the fragments' own layout.  (The
// warp-specialised kernel's form; RAW = false compiles the unrotated path out.)
template <int kWarps>
struct QueryLoads {
  float4 u0[kQ4NG / kWarps], u1[kQ4NG / kWarps];  // the thread's 8 values of each of its groups
};

template <int kWarps, bool RAW = true>
__device__ __forceinline__ void q4_query_load(const DecodeArgs& a, int b, int kvh, int warp, int lane,
                                              QueryLoads<kWarps>& L) {
  const int g = lane >> 2, t = lane & 3;
  // a column past the group reads head 0 (its fragments are zeroed)
  const int64_t row = ((int64_t)b * a.Hq + kvh * a.group + (g < a.group ? g : 0)) * kQ4D;
#pragma unroll
  for (int k = 0; k < kQ4NG / kWarps; ++k) {
    const int64_t e0 = row + 32 * (warp + kWarps * k) + 8 * t;
    if (RAW && a.q_raw != nullptr && a.q_dtype != KVQ_DT_F32) {  // 8 bf16 values: one 16-byte load
      const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(a.q_raw) + e0);
      L.u0[k] = make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                            __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
      L.u1[k] = make_float4(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u),
                            __uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u));
    } else {
      const float* src = RAW && a.q_raw != nullptr ? static_cast<const float*>(a.q_raw) : a.q;
      L.u0[k] = *reinterpret_cast<const float4*>(src + e0);
      L.u1[k] = *reinterpret_cast<const float4*>(src + e0 + 4);
    }
  }
}

template <int kWarps, bool RAW = true>
__device__ __forceinline__ void q4_query_build(const DecodeArgs& a, int warp, int lane, QueryLoads<kWarps>& L,
                                               uint4 (*qf)[2][32], float4 (*qb)[4]) {
  const int t = lane & 3;
  const bool live = (lane >> 2) < a.group;
  if (RAW && a.q_raw != nullptr && a.q_rotate) {
    // Rotate with the arithmetic of the rotation entry point: the fp32
    // butterfly, stages 1, 2, 4, 8, 16, (a, b) -> (a + b, a - b) with a the
    // lower index, then one multiply by fp32(1/sqrt(32)).  Stages 1, 2, 4 pair
    // the thread's own values; stages 8 and 16 pair threads t ^ 1 and t ^ 2 of
    // the same head (the same operands, so the same bits).
#pragma unroll
    for (int k = 0; k < kQ4NG / kWarps; ++k) {
      float x[8] = {L.u0[k].x, L.u0[k].y, L.u0[k].z, L.u0[k].w, L.u1[k].x, L.u1[k].y, L.u1[k].z, L.u1[k].w};
#pragma unroll
      for (int h = 1; h < 8; h <<= 1)
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if ((i & h) == 0) {
            const float lo = x[i], hi = x[i + h];
            x[i] = __fadd_rn(lo, hi);
            x[i + h] = __fsub_rn(lo, hi);
          }
#pragma unroll
      for (int m = 1; m <= 2; m <<= 1) {
        const bool upper = (t & m) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float o = __shfl_xor_sync(0xffffffffu, x[i], m);
          x[i] = upper ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(x[i], kHadamardScale);
      L.u0[k] = make_float4(x[0], x[1], x[2], x[3]);
      L.u1[k] = make_float4(x[4], x[5], x[6], x[7]);
    }
  }
  q4_frag_build<kWarps>(L.u0, L.u1, live, a.qscale, warp, lane, qf, qb);
  __syncthreads();
}

// ---------------------------------------------------------------- TQ4 rows
// A TQ4 code nibble is sign (bit 3) and magnitude index m (bits 0-2) of the
// level +-M_m of the 16-level Lloyd-Max codebook; the fp16 bits of M_0..M_7 are
// 0x301c 0x3635 0x3941 0x3b8a 0x3d06 0x3e79 0x4023 0x4177.  Byte tables of
// their low and high bytes, for prmt lookups indexed by m.
constexpr uint32_t kTqLo0 = 0x8a41351cu, kTqLo1 = 0x77237906u;  // low bytes of M_0..M_3, M_4..M_7
constexpr uint32_t kTqHi0 = 0x3b393630u, kTqHi1 = 0x41403e3du;  // high bytes

// The 8 codes of w (element i in nibble i: element 2b in the low nibble of
// byte b) -> 4 f16 pairs (elements 0,1 | 2,3 | 4,5 | 6,7), exactly the codebook
// levels.  The magnitudes select the levels' low and high bytes (prmt reads the
// low 16 bits of its selector: four 3-bit indices once the signs are masked);
// the signs are spread from bit 3 of each nibble to bit 7 of each high byte
// before the bytes are interleaved into pairs.
__device__ __forceinline__ uint4 tq4_levels8(uint32_t w) {
  const uint32_t mm = w & 0x77777777u;  // magnitudes of codes 0-3 (low half), 4-7 (high half)
  const uint32_t lo0 = prmt(kTqLo0, kTqLo1, mm), hi0s = prmt(kTqHi0, kTqHi1, mm);
  const uint32_t lo1 = prmt(kTqLo0, kTqLo1, mm >> 16), hi1s = prmt(kTqHi0, kTqHi1, mm >> 16);
  // x = w << 4 holds the signs of codes 0, 2, 4, 6 at bit 7 of its bytes 0-3;
  // w itself those of codes 1, 3, 5, 7
  const uint32_t x = w << 4;
  const uint32_t hi0 = hi0s ^ (prmt(x, w, 0x5140u) & 0x80808080u);  // codes 0, 1, 2, 3
  const uint32_t hi1 = hi1s ^ (prmt(x, w, 0x7362u) & 0x80808080u);  // codes 4, 5, 6, 7
  uint4 r;
  r.x = prmt(lo0, hi0, 0x5140u);  // (low, high) bytes of codes 0, 1
  r.y = prmt(lo0, hi0, 0x7362u);
  r.z = prmt(lo1, hi1, 0x5140u);
  r.w = prmt(lo1, hi1, 0x7362u);
  return r;
}

__device__ __forceinline__ float lds16h(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return __half2float(__ushort_as_half(v));
}

// TQ4 query fragments of one column tile: column g faces `qrow`; group G's
// fragment of lane (g, t) holds q[32G + 8t .. 8t + 7] (pairs in order), split
// into f16 high and low parts.  No bias: the levels enter signed.
template <int kWarps>
__device__ __forceinline__ void tq4_frag_prep(const float* qrow, bool live, float qscale, int warp, int lane,
                                              uint4 (*qf)[2][32]) {
  const int t = lane & 3;
  const float s = live ? qscale : 0.f;
#pragma unroll
  for (int k = 0; k < kQ4NG / kWarps; ++k) {
    const int G = warp + kWarps * k;
    const float4 u0 = *reinterpret_cast<const float4*>(qrow + 32 * G + 8 * t);
    const float4 u1 = *reinterpret_cast<const float4*>(qrow + 32 * G + 8 * t + 4);
    uint4 hi, lo;
    split_f16(u0.x * s, u0.y * s, hi.x, lo.x);
    split_f16(u0.z * s, u0.w * s, hi.y, lo.y);
    split_f16(u1.x * s, u1.y * s, hi.z, lo.z);
    split_f16(u1.z * s, u1.w * s, hi.w, lo.w);
    qf[G][0][lane] = hi;
    qf[G][1][lane] = lo;
  }
}

namespace q4r {

constexpr int kQ4Warps = 4;                       // warps per CTA = value group pairs in P.V
constexpr int kQ4TPW = 2;                         // 16-key tiles each warp scores per round
constexpr int kQ4RoundTiles = kQ4Warps * kQ4TPW;  // 8 tiles = 128 keys per round
constexpr int kQ4MaxColTiles = 4;                 // a decode window stacks up to 32 (row, head) columns
constexpr int kQ4GatherPart = 512;                // entries per partition of a gather (as the dense keys)

// Resident CTAs per SM the register budget is sized for: one column tile (one
// sequence's GQA group) fits 128 registers; each further tile adds 16 P.V
// accumulators per thread.
__host__ __device__ constexpr int q4_min_blocks(int nt) { return nt == 1 ? 4 : nt == 2 ? 3 : 2; }

// Warp w scores the round's tiles 2w, 2w + 1 and runs P.V for the value groups
// 2w, 2w + 1.  VR: rounds the V ring holds (1, or 2 where shared memory allows:
// round r + 1's V is then copied while round r is computed, with no wait for
// the warps to finish round r's P.V).
template <int NT, bool GATHER, int VR = 1>
struct __align__(1024) Q4Smem {
  static constexpr int kTile = q4_tile_bytes<GATHER>();
  uint8_t kc[kQ4Warps][kQ4TPW][kTile];         // K codes of each warp's tiles of the round (1024-aligned)
  uint8_t vc[VR][kQ4RoundTiles][kTile];        // V codes of the round's tiles, by round mod VR
  uint16_t ks[kQ4Warps][kQ4TPW][16 * 8];       // K scales
  uint16_t vs[VR][kQ4RoundTiles][16 * 8];      // V scales
  uint4 qf[NT][kQ4NG][2][32];                  // query fragments [column tile][group][hi, lo][lane]
  float4 qb[NT][kQ4NG][4];  // [column tile][group][t]: minus the code-offset bias of columns (2t, 2t+1, 2t, 2t+1)
  uint2 pb[kQ4RoundTiles][NT][32];  // [tile][column tile][lane]: P of the round as B fragments (keys 2t.., 2t+8..)
  float red[kQ4Warps][8 * NT];      // [warp][column]: maxima of each warp's tiles of the round
  float zs[kQ4RoundTiles][8 * NT];  // [tile slot][column]: sums of the probabilities of each slot's tiles
  uint64_t kbar[kQ4Warps];          // a warp's K tiles landed (kQ4TPW arrivals)
  uint64_t vfull[VR];               // the round's V tiles landed (kQ4RoundTiles arrivals)
  uint64_t vempty;                  // VR = 1: every warp is done with the round's V (kQ4Warps arrivals)
  int32_t grow[GATHER ? kQ4GatherPart : 1];  // gather: the cache row of each of the partition's entries
  int poison;
  int last;  // fused merge: this CTA finished its (sequence, KV head) last
};
// The unrotated-query path of the round kernel rotates the group's queries (8
// heads x 256 fp32) into V tiles 0..3, which are first filled after the prologue.
static_assert(sizeof(float) * 8 * kQ4D <= kQ4RoundTiles / 2 * kQ4TileBytes, "rotated queries fit vc[0..3]");

__device__ __forceinline__ void bar_sync_cta() { asm volatile("bar.sync 1, %0;" ::"n"(kQ4Warps * 32) : "memory"); }

// Issue the code copy of one dense 16-key tile of one plane (the scales come by
// the caller's lanes through the load path).  `row0` is the cache row of the
// tile's first key, computed ahead by the caller; < 0 (a bad page): no copy,
// and false (the tile then counts as poisoned; the barrier still gets this
// arrival so that nobody waits on it).
__device__ __forceinline__ bool q4_issue_plane(int32_t row0, const CUtensorMap* map, uint8_t* dc, uint64_t* bar) {
  if (row0 < 0) {
    mbar_arrive(bar);
    return false;
  }
  mbar_arrive_expect_tx(bar, kQ4TileBytes);
  tma_rows_2d(dc, map, row0, bar);
  return true;
}

// The calling warp's TPW tiles of round `rd` of one plane into dc[u], ds[u]
// (dense: lane 0 issues the code copies, 16 lanes a tile the scales; gather:
// every lane copies rows).  A tile past the partition still arrives on `bar`.
// Returns true for a tile with a bad page or index.
template <bool GATHER, bool TQ = false, int TPW = 2>
__device__ __forceinline__ bool q4_issue_own(const DecodeArgs& a, int b, int kvh, int k0, int k1, int rd, int warp,
                                             int lane, int32_t tile_row, const int32_t* grow, const CUtensorMap* map,
                                             const void* codes, const void* scales,
                                             uint8_t (*dc)[q4_tile_bytes<GATHER>()], uint16_t (*ds)[16 * 8],
                                             uint64_t* bar) {
  const int tile0 = kQ4RoundTiles * rd + TPW * warp;
  if constexpr (GATHER) {
    // grow[i]: the cache row of the partition's entry i (-1: a bad index or
    // page, already flagged).  The warp copies its tiles' rows through the load
    // path, 16 bytes a lane (a row's 128 code bytes by 8 lanes, 4 rows per
    // instruction; the 16 scale bytes of row l by lane l): one bulk copy per row
    // would queue 32 requests a tile on the copy engine.  Each lane's copies are
    // tracked on the barrier before lane 0's arrival for each tile.
    bool bad = false;
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const int e0 = 16 * (tile0 + u);  // the tile's first entry in the partition
      const int nvalid = min(16, k1 - k0 - e0);
      if (nvalid <= 0) continue;  // warp-uniform
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int c = lane + 32 * x, r = c >> 3, part = c & 7;
        const int32_t row = r < nvalid ? grow[e0 + r] : -1;
        if (row >= 0)
          cp_async_16(dc[u] + r * kQ4GatherRow + 16 * part, static_cast<const uint8_t*>(codes) + (int64_t)row * 128 + 16 * part);
      }
      const int32_t srow = lane < nvalid ? grow[e0 + lane] : -1;
      if (lane < 16 && srow >= 0)
        cp_async_16(ds[u] + 8 * lane, static_cast<const uint16_t*>(scales) + (int64_t)srow * 8);
      bad |= __any_sync(0xffffffffu, lane < nvalid && srow < 0);
    }
    cp_async_mbar_track(bar);
    __syncwarp();
    if (lane == 0)
#pragma unroll
      for (int u = 0; u < TPW; ++u) mbar_arrive(bar);
    return bad;
  } else {
    int32_t rows[TPW];
#pragma unroll
    for (int u = 0; u < TPW; ++u) rows[u] = __shfl_sync(0xffffffffu, tile_row, (tile0 + u) & 31);
    bool bad = false;
    // A dense tile's scales (16 consecutive rows: 256 bytes, TQ4 32) by 16-byte
    // cp.async through the load path, lanes 16u .. of tile u, so that the copy
    // engine, which takes its requests one after another, gets one per tile
    // (the codes); each lane's copy is tracked on the tile's barrier before the
    // tile's arrival below can complete the phase.
    static_assert(TPW <= 2, "16 lanes per tile's scales");
    constexpr int kScaleLanes = (TQ ? 32 : kQ4ScaleBytes) / 16;
    const int u = lane >> 4, part = lane & 15;
    int32_t row = rows[0];  // rows[u], without indexing the array by a lane-dependent value
#pragma unroll
    for (int v = 1; v < TPW; ++v)
      if (u == v) row = rows[v];
    if (u < TPW && part < kScaleLanes && k0 + 16 * (tile0 + u) < k1 && row >= 0) {
      const uint16_t* src = static_cast<const uint16_t*>(scales) + (int64_t)row * (TQ ? 1 : 8) + 8 * part;
      cp_async_16(&ds[0][0] + 16 * 8 * u + 8 * part, src);
      cp_async_mbar_track(bar);
    }
    __syncwarp();
    if (lane == 0) {
      fence_proxy_async();  // the buffers were last read through the generic proxy
#pragma unroll
      for (int u = 0; u < TPW; ++u) {
        const int key0 = k0 + 16 * (tile0 + u);
        if (key0 >= k1)
          mbar_arrive(bar);
        else if (!q4_issue_plane(rows[u], map, dc[u], bar))
          bad = true;
      }
    }
    return bad;
  }
}

// The fused merge (kvq_decode_merged) folds partials in two levels: the last
// CTA of each block of kMergeBlock consecutive partitions of a (sequence b,
// KV head) folds that block's partials into a block partial, and the last of
// the group's block folders folds the block partials into the outputs.  The
// tree depends only on the partition indices, so the outputs do not depend on
// the batch or on which CTA finishes last.
constexpr int kQ4FoldCols = 4;  // 4-dim columns per thread in a fold: 8 heads x 64 / 128 threads

// Loads entries i .. i + 3 of a fold thread's columns (column k at ap[k]).
__device__ __forceinline__ void q4_fold_load(float4 (&v)[kQ4FoldCols][4], const float* const (&ap)[kQ4FoldCols],
                                             int t, int ncol, int i) {
#pragma unroll
  for (int k = 0; k < kQ4FoldCols; ++k)
    if (t + k * kQ4Warps * 32 < ncol)
#pragma unroll
      for (int u = 0; u < 4; ++u) v[k][u] = __ldcg(reinterpret_cast<const float4*>(ap[k] + (int64_t)(i + u) * kQ4D));
}

// Fold n entries (i ascending) of each of the group's heads: M = max m_i,
// w_i = 2^(m_i - M), Z = sum z_i w_i, acc = sum acc_i w_i.  Entry i of head h
// sits at m[h * hs + i], z[h * hs + i], acc[(h * hs + i) * 256 ..].  Warp w
// computes the weights of heads 2w and 2w + 1 together (lanes over i; the m_i
// stashed in wts by the first pass, the z_i read in the second; Z by a fixed
// xor tree).  Then thread t takes the 4-dim columns t, t + 128, .. of the
// group (column c: head c / 64, dims 4 (c % 64) ..) and loads four entries of
// each of its columns at a time; every output is one fused multiply-add chain
// over i ascending.  final = false: (M, Z, acc) go to om, oz, oacc at
// [h * ohs] (M = NaN if some m_i is NaN); final = true: out = acc / Z (0 for a
// group without keys, NaN for a NaN), rotated back per 32-group when
// rotate_back, at out + h * 256.
__device__ __forceinline__ void q4_fold(const float* m, const float* z, const float* acc, int64_t hs, int n,
                                        int group, float* wts, float* zsum, bool final, float* om, float* oz,
                                        float* oacc, int64_t ohs, float* out, bool rotate_back) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float* mx = zsum + 8;  // [group]: the heads' maxima
  const int ncol = group * (kQ4D / 4);
  const int t = threadIdx.x;
  const float* ap[kQ4FoldCols];
  int hc[kQ4FoldCols];
  float4 o[kQ4FoldCols];
#pragma unroll
  for (int k = 0; k < kQ4FoldCols; ++k) {
    const int c = t + k * kQ4Warps * 32;
    hc[k] = c >> 6;
    ap[k] = acc + hc[k] * hs * kQ4D + 4 * (c & 63);
    o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // the first four entries' loads overlap the weights
  float4 v[kQ4FoldCols][4];
  if (n >= 4) q4_fold_load(v, ap, t, ncol, 0);
  const int ha = 2 * warp, hb = 2 * warp + 1;
  if (ha < group) {
    const bool two = hb < group;
    float Ma = -INFINITY, Mb = -INFINITY;
    bool nan_a = false, nan_b = false;
#pragma unroll 4
    for (int i = lane; i < n; i += 32) {
      const float va = __ldcg(m + ha * hs + i);
      const float vb = two ? __ldcg(m + hb * hs + i) : -INFINITY;
      wts[ha * n + i] = va;
      if (two) wts[hb * n + i] = vb;
      nan_a |= isnan(va);
      nan_b |= isnan(vb);
      Ma = fmaxf(Ma, va);
      Mb = fmaxf(Mb, vb);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Ma = fmaxf(Ma, __shfl_xor_sync(0xffffffffu, Ma, o));
      Mb = fmaxf(Mb, __shfl_xor_sync(0xffffffffu, Mb, o));
    }
    nan_a = __any_sync(0xffffffffu, nan_a);
    nan_b = __any_sync(0xffffffffu, nan_b);
    float Za = 0.f, Zb = 0.f;
#pragma unroll 4
    for (int i = lane; i < n; i += 32) {
      const float za = __ldcg(z + ha * hs + i);
      const float zb = two ? __ldcg(z + hb * hs + i) : 0.f;
      const float wa = (Ma == -INFINITY) ? 0.f : exp2f(wts[ha * n + i] - Ma);
      wts[ha * n + i] = wa;
      Za = fmaf(za, wa, Za);
      if (two) {
        const float wb = (Mb == -INFINITY) ? 0.f : exp2f(wts[hb * n + i] - Mb);
        wts[hb * n + i] = wb;
        Zb = fmaf(zb, wb, Zb);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      Za += __shfl_xor_sync(0xffffffffu, Za, o);
      Zb += __shfl_xor_sync(0xffffffffu, Zb, o);
    }
    if (lane == 0) {
      zsum[ha] = nan_a ? NAN : Za;
      mx[ha] = nan_a ? NAN : Ma;
      if (two) {
        zsum[hb] = nan_b ? NAN : Zb;
        mx[hb] = nan_b ? NAN : Mb;
      }
    }
  }
  __syncthreads();
  int i = 0;
  for (; i + 4 <= n; i += 4) {  // four entries of every column in flight
    if (i > 0) q4_fold_load(v, ap, t, ncol, i);
#pragma unroll
    for (int k = 0; k < kQ4FoldCols; ++k)
      if (t + k * kQ4Warps * 32 < ncol)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float w = wts[hc[k] * n + i + u];
          o[k].x = fmaf(v[k][u].x, w, o[k].x);
          o[k].y = fmaf(v[k][u].y, w, o[k].y);
          o[k].z = fmaf(v[k][u].z, w, o[k].z);
          o[k].w = fmaf(v[k][u].w, w, o[k].w);
        }
  }
  for (; i < n; ++i) {
#pragma unroll
    for (int k = 0; k < kQ4FoldCols; ++k)
      if (t + k * kQ4Warps * 32 < ncol) {
        const float4 vi = __ldcg(reinterpret_cast<const float4*>(ap[k] + (int64_t)i * kQ4D));
        const float w = wts[hc[k] * n + i];
        o[k].x = fmaf(vi.x, w, o[k].x);
        o[k].y = fmaf(vi.y, w, o[k].y);
        o[k].z = fmaf(vi.z, w, o[k].z);
        o[k].w = fmaf(vi.w, w, o[k].w);
      }
  }
  if (!final) {
#pragma unroll
    for (int k = 0; k < kQ4FoldCols; ++k) {
      const int c = t + k * kQ4Warps * 32;
      if (c < ncol) *reinterpret_cast<float4*>(oacc + hc[k] * ohs * kQ4D + 4 * (c & 63)) = o[k];
    }
    if (t < group) {
      om[t * ohs] = mx[t];
      oz[t * ohs] = zsum[t];
    }
    return;
  }
#pragma unroll
  for (int k = 0; k < kQ4FoldCols; ++k) {
    const int c = t + k * kQ4Warps * 32;
    if (c >= ncol) continue;  // warp-uniform: ncol is a multiple of 64
    const float Z = zsum[hc[k]];
    const bool empty = !(Z > 0.f) && !isnan(Z);
    float x0 = empty ? 0.f : o[k].x / Z, x1 = empty ? 0.f : o[k].y / Z;
    float x2 = empty ? 0.f : o[k].z / Z, x3 = empty ? 0.f : o[k].w / Z;
    if (rotate_back) {
      // 32-point butterfly of the group, stages by dim bit 0 .. 4: bits 0, 1
      // within the thread's 4 dims, bits 2 .. 4 across lanes (lane bits 0 .. 2);
      // the lower element takes lower + upper, the upper lower - upper
      const float a0 = x0 + x1, a1 = x0 - x1, a2 = x2 + x3, a3 = x2 - x3;
      float b[4] = {a0 + a2, a1 + a3, a0 - a2, a1 - a3};
#pragma unroll
      for (int o2 = 1; o2 < 8; o2 <<= 1) {
        const bool upper = (lane & o2) != 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p = __shfl_xor_sync(0xffffffffu, b[j], o2);
          b[j] = upper ? p - b[j] : b[j] + p;
        }
      }
      x0 = __fmul_rn(b[0], kHadamardScale);
      x1 = __fmul_rn(b[1], kHadamardScale);
      x2 = __fmul_rn(b[2], kHadamardScale);
      x3 = __fmul_rn(b[3], kHadamardScale);
    }
    *reinterpret_cast<float4*>(out + hc[k] * kQ4D + 4 * (c & 63)) = make_float4(x0, x1, x2, x3);
  }
}

// Byte offset of this lane's ldmatrix row address for group-chunk G (+ lane >> 4)
// inside a code tile (see the kernel's fragment layout).  Dense tiles carry the
// 128-byte swizzle (chunk c of row r at c ^ (r & 7)); gather tiles are padded rows.
template <bool GATHER>
__device__ __forceinline__ uint32_t q4_chunk_off(int lrow, int lhi, int lane, int G) {
  return GATHER ? lrow * kQ4GatherRow + ((G + lhi) << 4) : lrow * 128 + (((G + lhi) ^ (lane & 7)) << 4);
}

constexpr uint32_t kQfTileBytes = kQ4NG * 2 * 32 * 16;  // query fragments of one column tile
constexpr uint32_t kQbTileBytes = kQ4NG * 4 * 16;       // query biases of one column tile

// Scores of a warp's TPW tiles of a round (4-bit rows, not TQ4): S[u][nt][.] +=
// the scaled dot products of keys g, g + 8 of tile u with columns 2t, 2t + 1 of
// column tile nt (S enters as zeros).  The K codes of tile u sit at kc_base + u *
// tile bytes, its scales at ks_base + u * 256; the query fragments and biases at
// qf_addr / qb_addr (this lane's entries of column tile 0).
template <bool GATHER, int NT, int TPW>
__device__ __forceinline__ void q4_score_tiles(float (&S)[TPW][NT][4], uint32_t kc_base, uint32_t ks_base,
                                               uint32_t qf_addr, uint32_t qb_addr, int lrow, int lhi, int lane) {
  const int g = lane >> 2;
#pragma unroll
  for (int w = 0; w < kQ4NG / 2; ++w) {  // group pair (2w, 2w+1): one word of each fragment row
    // kw[u]: codes 8t .. 8t+7 of group 2w (.x key g, .y key g+8) and of group 2w+1 (.z, .w)
    uint4 kw[TPW];
    float2 fsa[TPW], fsb[TPW];
    const uint32_t okl = q4_chunk_off<GATHER>(lrow, lhi, lane, 2 * w);
#pragma unroll
    for (int u = 0; u < TPW; ++u) {
      const uint32_t kb = kc_base + u * q4_tile_bytes<GATHER>(), sb = ks_base + u * kQ4ScaleBytes;
      kw[u] = ldsm_x4(kb + okl);
      fsa[u] = __half22float2(u32_as_h2(lds32a(sb + g * 16 + 4 * w)));  // K scales (2w, 2w+1) of row g
      fsb[u] = __half22float2(u32_as_h2(lds32a(sb + (g + 8) * 16 + 4 * w)));
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int G = 2 * w + e;
      uint4 qh[NT], ql[NT];
      float4 nb[NT];  // -bias of columns (2t, 2t+1, 2t, 2t+1)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        qh[nt] = lds128a(qf_addr + nt * kQfTileBytes + G * 1024);
        ql[nt] = lds128a(qf_addr + nt * kQfTileBytes + G * 1024 + 512);
        nb[nt] = lds128f(qb_addr + nt * kQbTileBytes + G * 64);
      }
#pragma unroll
      for (int u = 0; u < TPW; ++u) {
        // codes 8t .. 8t+7 of keys g (xa1) and g+8 (xb1); the nibble pairs
        // (0, 4), (1, 5) sit in bits 0-3 / 16-19 and 4-7 / 20-23; shifted by a
        // byte (xa2, xb2), the pairs (2, 6), (3, 7)
        const uint32_t xa1 = e ? kw[u].z : kw[u].x, xb1 = e ? kw[u].w : kw[u].y;
        const uint32_t xa2 = xa1 >> 8, xb2 = xb1 >> 8;
        const uint32_t a10 = nib_lo_pair_biased(xa1), a11 = nib_lo_pair_biased(xb1);
        const uint32_t a12 = nib_hi_pair_biased(xa1), a13 = nib_hi_pair_biased(xb1);
        const uint32_t a20 = nib_lo_pair_biased(xa2), a21 = nib_lo_pair_biased(xb2);
        const uint32_t a22 = nib_hi_pair_biased(xa2), a23 = nib_hi_pair_biased(xb2);
        const float sa = e ? fsa[u].y : fsa[u].x, sb = e ? fsb[u].y : fsb[u].x;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float part[4];
          mma_f16_c(part, a10, a11, a12, a13, qh[nt].x, qh[nt].y, nb[nt].x, nb[nt].y, nb[nt].z, nb[nt].w);
          mma_f16(part, a20, a21, a22, a23, qh[nt].z, qh[nt].w);
          mma_f16(part, a10, a11, a12, a13, ql[nt].x, ql[nt].y);
          mma_f16(part, a20, a21, a22, a23, ql[nt].z, ql[nt].w);
          S[u][nt][0] = fmaf(sa, part[0], S[u][nt][0]);
          S[u][nt][1] = fmaf(sa, part[1], S[u][nt][1]);
          S[u][nt][2] = fmaf(sb, part[2], S[u][nt][2]);
          S[u][nt][3] = fmaf(sb, part[3], S[u][nt][3]);
        }
      }
    }
  }
}

// P.V of one round (4-bit rows, not TQ4): acc[e][.][nt] += the warp's value
// groups 2w + e of the round's 8 tiles times their probabilities.  pb_addr:
// this lane's B fragment of tile 0 (tiles 256 * NT bytes apart); vc_base,
// vs_base: the round's V codes (tile j at + j * tile bytes) and the scale word of
// the warp's groups; off_vl: the lane's ldmatrix offset of their chunks; kr0:
// the round's first key, k1: the partition's end (kTail: zero the V scales of
// keys at or past k1, so their stale codes add nothing).
template <bool kTail, bool GATHER, int NT>
__device__ __forceinline__ void q4_pv_tiles(float (&acc)[2][2][NT][4], uint32_t pb_addr, uint32_t vc_base,
                                            uint32_t vs_base, uint32_t off_vl, int kr0, int k1, int lane) {
  const int t = lane & 3;
#pragma unroll
  for (int j = 0; j < kQ4RoundTiles; ++j) {
    uint2 pp[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) pp[nt] = lds64a(pb_addr + (j * NT + nt) * 256);
    const uint32_t cb = vc_base + j * q4_tile_bytes<GATHER>();
    const uint32_t sb = vs_base + j * kQ4ScaleBytes;
    // V scales of keys 2t, 2t+1, 2t+8, 2t+9 and V codes of the same rows:
    // codes 4g .. 4g+3 of groups 2w, 2w+1 (ldmatrix, transposed).
    uint32_t swa = lds32a(sb + (2 * t) * 16);
    uint32_t swb = lds32a(sb + (2 * t + 1) * 16);
    uint32_t swc = lds32a(sb + (2 * t + 8) * 16);
    uint32_t swd = lds32a(sb + (2 * t + 9) * 16);
    if constexpr (kTail) {
      const int nvalid = k1 - (kr0 + 16 * j);
      if (nvalid < 16) {  // CTA-uniform
        if (2 * t >= nvalid) swa = 0u;
        if (2 * t + 1 >= nvalid) swb = 0u;
        if (2 * t + 8 >= nvalid) swc = 0u;
        if (2 * t + 9 >= nvalid) swd = 0u;
      }
    }
    // .x: keys 2t, 2t+1 of group 2w (bytes 2g, 2g+1 of each key, key 2t in the low
    // half), .y: keys 2t+8, 2t+9; .z, .w: group 2w+1
    const uint4 vw = ldsm_x4_trans(cb + off_vl);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const uint32_t ssel = e ? 0x7632u : 0x5410u;
      const uint32_t slo = prmt(swa, swb, ssel);
      const uint32_t shi = prmt(swc, swd, ssel);
      const uint32_t x01 = e ? vw.z : vw.x;  // codes 4g, 4g+1 in the low byte of each half
      const uint32_t x23 = e ? vw.w : vw.y;
      const uint32_t x01b = x01 >> 8, x23b = x23 >> 8;  // codes 4g+2, 4g+3
      // d-tile (G,0): rows g <-> d = 32G+4g, g+8 <-> 32G+4g+2 ; (G,1): +1
      const uint32_t l0 = nib_lo_pair(x01), l1 = nib_lo_pair(x01b), l2 = nib_lo_pair(x23), l3 = nib_lo_pair(x23b);
      const uint32_t h0 = nib_hi_pair(x01), h1 = nib_hi_pair(x01b), h2 = nib_hi_pair(x23), h3 = nib_hi_pair(x23b);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const uint32_t b0 = h2_as_u32(__hmul2(u32_as_h2(pp[nt].x), u32_as_h2(slo)));
        const uint32_t b1 = h2_as_u32(__hmul2(u32_as_h2(pp[nt].y), u32_as_h2(shi)));
        mma_f16(acc[e][0][nt], l0, l1, l2, l3, b0, b1);
        mma_f16(acc[e][1][nt], h0, h1, h2, h3, b0, b1);
      }
    }
  }
}

// kvq_decode_step: the CTA whose partition holds sequence b's new position pos
// stores the new K and V rows of KV head kvh there -- the warps take the (plane,
// group) pairs in turn, each with the warp-level group code of the store kernels
// (the same bits as kvq_store) -- before it issues any tile copy.  The writes are
// fenced for the async proxy, and the CTA barrier orders them before the copies
// that read them back.  A bad page writes nothing (the tile's own check flags
// and poisons it).
__device__ __forceinline__ void q4_store_new_token(const DecodeArgs& a, int b, int kvh, int32_t pos, int warp,
                                                   int lane, int nwarps) {
  const kvq_cache& c = a.c;
  const int32_t page = a.block_tables[(int64_t)b * a.bt_stride + pos / c.page_size];
  if (page >= 0 && page < c.num_pages) {
    const int64_t row = ((int64_t)page * c.num_kv_heads + kvh) * c.page_size + pos % c.page_size;
    const int64_t src = ((int64_t)b * c.num_kv_heads + kvh) * kQ4D + lane;
    const bool rot = c.format == KVQ_FMT_Q4_HAD32;
    for (int task = warp; task < 2 * kQ4NG; task += nwarps) {  // warp-uniform
      const int plane = task >= kQ4NG ? 1 : 0, G = task - plane * kQ4NG;
      const float x = load_act(plane ? a.new_v : a.new_k, a.new_dtype, src + 32 * G);
      __half s16;
      const uint32_t code = rot ? q4_group_code_warp<true>(x, lane, s16) : q4_group_code_warp<false>(x, lane, s16);
      q4_write_group_warp(static_cast<uint8_t*>(plane ? c.v : c.k) + row * (kQ4D / 2),
                          static_cast<uint16_t*>(plane ? c.v_scale : c.k_scale) + row * kQ4NG, G, code, s16, lane);
    }
    fence_proxy_async_global();
  }
  __syncthreads();
}

// One CTA per (partition, KV head, column set).  NT column tiles of 8 columns
// face the keys on the MMA's N side.  A plain decode (WIN = false, NT = 1) gives
// the columns to the heads of one sequence's GQA group.  A decode window
// (WIN = true) gives them to (row, head) pairs of `rows_per_cta` rows of one
// sequence, row-major: the rows share the block table and so every key, whose
// codes are then converted once for all of them; each row keeps its own causal
// end (its length), its own softmax state and its own partials.
// MINB: resident CTAs per SM the registers are budgeted for (0: q4_min_blocks);
// the fused merge on a grid that fits in two CTAs per SM takes MINB = 2 (up to
// 255 registers) and VR = 2 (a two-round V ring).  The arithmetic is the same
// either way; only the copy schedule differs.
template <bool GATHER, int NT, bool WIN, bool TQ = false, bool LM = false, int MINB = 0, int VR = 1>
__global__ void __launch_bounds__(kQ4Warps * 32, MINB ? MINB : q4_min_blocks(NT))
    decode_q4_round_kernel(const __grid_constant__ DecodeArgs a) {
  static_assert(!(WIN && GATHER), "decode windows read dense prefixes");
  static_assert(WIN || NT == 1, "one sequence's group fills one column tile");
  static_assert(!TQ || (!GATHER && !WIN), "TQ4 rows: dense single-sequence decode");
  static_assert(!LM || (!GATHER && !WIN && !TQ), "the fused merge: dense 4-bit decode");
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles (the launch adds 1 KB of slack)
  Q4Smem<NT, GATHER, VR>& sm =
      *reinterpret_cast<Q4Smem<NT, GATHER, VR>*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  constexpr int kTile = q4_tile_bytes<GATHER>();
  const int p = blockIdx.x, kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  // rows [b, b + nr): one sequence, or a slice of a window's rows
  const int b = WIN ? blockIdx.z * a.rows_per_cta : blockIdx.z;
  const int nr = WIN ? min(a.rows_per_cta, a.nrows - b) : 1;

  // Metadata first: the lengths and block tables are caller inputs that no
  // kernel of this library writes, so they are read before the wait on the
  // previous kernel of the stream (programmatic dependent launch) and their
  // latency overlaps it.  The cache, the queries and every write come after.
  int32_t T;                // keys of the CTA's longest row
  int32_t Tmin = 0;         // window: keys of its shortest row (a bad row counts 0)
  int32_t row_len = 0;      // window: lane i < nr holds the length of row b + i
  bool bad_len = false;     // plain: the sequence's length is invalid
  bool bad_row = false;     // window: some row's length is invalid (that row is skipped)
  if (GATHER) {
    T = a.n_sel;
  } else if (!WIN) {
    T = a.seq_lens[b];
    bad_len = T < 0 || T > a.max_seq_len || (int64_t)T > (int64_t)a.max_pages * a.c.page_size;
  } else {
    bool bad = false;
    if (lane < nr) {
      row_len = a.seq_lens[b + lane];
      bad = row_len < 0 || row_len > a.max_seq_len || (int64_t)row_len > (int64_t)a.max_pages * a.c.page_size;
      if (bad) row_len = 0;
    }
    bad_row = __any_sync(0xffffffffu, bad);
    T = row_len;
    Tmin = lane < nr ? row_len : INT32_MAX;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T = max(T, __shfl_xor_sync(0xffffffffu, T, o));
      Tmin = min(Tmin, __shfl_xor_sync(0xffffffffu, Tmin, o));
    }
  }
  const int nparts = bad_len ? 0 : (T + a.part - 1) / a.part;
  const bool active = p < nparts;  // CTA-uniform
  const int k0 = p * a.part;
  const int k1 = min(k0 + a.part, T);
  const int ntiles = active ? (k1 - k0 + 15) / 16 : 0;
  const int nrounds = (ntiles + kQ4RoundTiles - 1) / kQ4RoundTiles;  // <= 4
  // tile u of warp w in round r: kQ4RoundTiles * r + kQ4TPW * w + u

  // Window: the length of the row of each of this thread's score columns
  // (columns 8 nt + 2t + c); a column past the CTA's rows takes T.
  int32_t colen[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int row = (8 * nt + 2 * t + c) / a.group;
      const int32_t len = __shfl_sync(0xffffffffu, row_len, row & 31);
      colen[nt][c] = row < nr ? len : T;
    }

  // Lane i: the cache row of tile i (its first key), computed once so that the
  // copies need neither a global load nor a division inside the loop; -1 for a
  // bad page.
  int32_t tile_row = -1;
  bool bad_page = false;
  if (!GATHER && lane < ntiles) {
    const int key0 = k0 + 16 * lane;
    const int32_t page = a.block_tables[(int64_t)b * a.bt_stride + key0 / a.c.page_size];
    if (page < 0 || page >= a.c.num_pages)
      bad_page = true;
    else
      tile_row = static_cast<int32_t>(((int64_t)page * a.c.num_kv_heads + kvh) * a.c.page_size + key0 % a.c.page_size);
  }
  if (active && threadIdx.x == 0) {
    for (int w = 0; w < kQ4Warps; ++w) mbar_init(&sm.kbar[w], kQ4TPW);
    for (int i = 0; i < VR; ++i) mbar_init(&sm.vfull[i], kQ4RoundTiles);
    mbar_init(&sm.vempty, kQ4Warps);
    sm.poison = 0;
    fence_barrier_init();
  }

  pdl_wait();
  if constexpr (LM) {
    // no partition will count in: partition 0's CTA writes the outputs itself
    // (NaN for an invalid length, zeros for an empty sequence)
    if ((bad_len || nparts == 0) && p == 0)
      for (int i = threadIdx.x; i < a.group * kQ4D; i += kQ4Warps * 32)
        a.fused_out[((int64_t)b * a.Hq + kvh * a.group) * kQ4D + i] = bad_len ? NAN : 0.f;
  }
  if (bad_len) {
    if (threadIdx.x == 0 && p == 0 && kvh == 0) set_status(a.status, KVQ_DEV_BAD_LENGTH);
    return;  // the merge writes NaN for this sequence
  }
  if (bad_row && threadIdx.x == 0 && p == 0 && kvh == 0) set_status(a.status, KVQ_DEV_BAD_LENGTH);
  if (!active) return;
  if (bad_page && warp == 0) set_status(a.status, KVQ_DEV_BAD_PAGE);
  __syncthreads();  // the mbarriers are initialised
  if constexpr (!GATHER && !WIN && !TQ) {
    if (a.new_k != nullptr && p == (T - 1) / a.part) q4_store_new_token(a, b, kvh, T - 1, warp, lane, kQ4Warps);
  }
  const int32_t* grow = nullptr;
  if constexpr (GATHER) {
    // The partition's selected rows, resolved once and in parallel (each is a
    // chain of two dependent loads: the selected position, then its page); an
    // index outside the sequence (or its block table) or a bad page is flagged
    // and its row poisons the tiles that hold it.
    const int32_t Tseq = a.seq_lens[b];
    const int32_t* bt = a.block_tables + (int64_t)b * a.bt_stride;
    const int64_t tmax = (int64_t)a.max_pages * a.c.page_size;
    for (int i = threadIdx.x; i < k1 - k0; i += kQ4Warps * 32) {
      const int32_t pos = a.sel[(int64_t)b * a.n_sel + k0 + i];
      int32_t row = -1;
      if (pos < 0 || pos >= Tseq || pos >= tmax) {
        set_status(a.status, KVQ_DEV_BAD_INDEX);
      } else {
        const int32_t pg = bt[pos / a.c.page_size];
        if (pg < 0 || pg >= a.c.num_pages)
          set_status(a.status, KVQ_DEV_BAD_PAGE);
        else
          row = static_cast<int32_t>(((int64_t)pg * a.c.num_kv_heads + kvh) * a.c.page_size + pos % a.c.page_size);
      }
      sm.grow[i] = row;
    }
    __syncthreads();
    grow = sm.grow;
  }

  const kvq_cache& c = a.c;
  bool poisoned = q4_issue_own<GATHER, TQ, kQ4TPW>(a, b, kvh, k0, k1, 0, warp, lane, tile_row, grow, &a.tm_k, c.k, c.k_scale,
                                       sm.kc[warp], sm.ks[warp], &sm.kbar[warp]);

  // V of round 0 (and 1), after the query fragments: the in-kernel rotation uses
  // vc[0][0..3] until the prologue's last barrier, and K(0), which the first
  // round waits for, goes out alone first
  auto issue_v01 = [&]() {
    poisoned |= q4_issue_own<GATHER, TQ, kQ4TPW>(a, b, kvh, k0, k1, 0, warp, lane, tile_row, grow, &a.tm_v, c.v, c.v_scale,
                                                 &sm.vc[0][kQ4TPW * warp], &sm.vs[0][kQ4TPW * warp], &sm.vfull[0]);
    if constexpr (VR == 2) {
      if (nrounds > 1)
        poisoned |= q4_issue_own<GATHER, TQ, kQ4TPW>(a, b, kvh, k0, k1, 1, warp, lane, tile_row, grow, &a.tm_v, c.v,
                                                     c.v_scale, &sm.vc[1][kQ4TPW * warp], &sm.vs[1][kQ4TPW * warp],
                                                     &sm.vfull[1]);
    }
  };

  if constexpr (WIN) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = 8 * nt + g, row = col / a.group;
      const bool live = row < nr;
      const float* qrow = a.q + ((int64_t)(b + (live ? row : 0)) * a.Hq + kvh * a.group + (live ? col - row * a.group : 0)) * kQ4D;
      q4_frag_prep<kQ4Warps>(qrow, live, a.qscale, warp, lane, sm.qf[nt], sm.qb[nt]);
    }
    __syncthreads();
  } else if constexpr (TQ) {
    const bool live = g < a.group;
    tq4_frag_prep<kQ4Warps>(a.q + ((int64_t)b * a.Hq + kvh * a.group + (live ? g : 0)) * kQ4D, live, a.qscale, warp,
                            lane, sm.qf[0]);
    __syncthreads();
  } else {
    q4r_query_prep<kQ4Warps>(a, b, kvh, warp, lane, reinterpret_cast<float*>(&sm.vc[0][0][0]), sm.qf[0], sm.qb[0]);
  }
  issue_v01();
  const uint32_t qf_addr = smem_u32(&sm.qf[0][0][0][lane]);
  const uint32_t qb_addr = smem_u32(&sm.qb[0][0][t]);

  // P.V accumulators of groups 2w + e, d-tiles (G, 0) and (G, 1), column tile nt
  float acc[2][2][NT][4];
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[e][j][nt][i] = 0.f;
  // running max of columns 2t, 2t+1 of each column tile (base 2), equal in every
  // warp, and this thread's partial sums of the probabilities, one per tile slot
  // u (the warp's tile u of every round), so that the sums are added in the same
  // order whatever the number of warps
  float m0[NT], m1[NT], z0[kQ4TPW][NT], z1[kQ4TPW][NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m0[nt] = m1[nt] = kQ4NoMax;
#pragma unroll
    for (int u = 0; u < kQ4TPW; ++u) z0[u][nt] = z1[u][nt] = 0.f;
  }
  bool timed_out = false;

  // ldmatrix addresses inside a code tile.  A row is 8 groups of 16 bytes (32
  // codes each); lane l addresses row (l & 7) + 8 ((l >> 3) & 1), group-chunk
  // G + (l >> 4), so the four matrices are (keys 0-7, G), (keys 8-15, G),
  // (keys 0-7, G + 1), (keys 8-15, G + 1).  Dense tiles carry the 128-byte
  // swizzle (chunk c of row r at c ^ (r & 7)); gather tiles are padded rows.
  const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lhi = lane >> 4;
  auto chunk_off = [&](int G) -> uint32_t { return q4_chunk_off<GATHER>(lrow, lhi, lane, G); };  // G even
  const uint32_t off_vl = chunk_off(2 * warp);  // V: groups 2w, 2w + 1 of this warp
  const uint32_t kc_base = smem_u32(&sm.kc[warp][0][0]);
  const uint32_t ks_base = smem_u32(&sm.ks[warp][0][0]);
  constexpr uint32_t kVcSlot = sizeof(sm.vc[0]), kVsSlot = sizeof(sm.vs[0]);
  const uint32_t pb_addr = smem_u32(&sm.pb[0][0][lane]);

  for (int r = 0; r < nrounds; ++r) {
    const uint32_t par = r & 1;
    const int tile0 = kQ4RoundTiles * r + kQ4TPW * warp;
    float S[kQ4TPW][NT][4];
#pragma unroll
    for (int u = 0; u < kQ4TPW; ++u)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) S[u][nt][0] = S[u][nt][1] = S[u][nt][2] = S[u][nt][3] = -INFINITY;
    if (k0 + 16 * tile0 < k1) {  // warp-uniform: this warp has at least one tile in the round
      // mma.sync below is warp-collective: the wait's outcome is made warp-uniform
      if (!timed_out && !__all_sync(0xffffffffu, mbar_wait_bounded(&sm.kbar[warp], par))) timed_out = true;

      // ---------------- scores S[u][nt][key][column] for keys g, g+8 of tile u and columns 2t, 2t+1
#pragma unroll
      for (int u = 0; u < kQ4TPW; ++u)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) S[u][nt][0] = S[u][nt][1] = S[u][nt][2] = S[u][nt][3] = 0.f;
      if constexpr (TQ) {
        // TQ4: the levels enter signed and exact; one accumulator chain over
        // all 8 groups, then the row's scale (keys g, g + 8).
#pragma unroll
        for (int w = 0; w < kQ4NG / 2; ++w) {
          uint4 kw[kQ4TPW];
          const uint32_t okl = chunk_off(2 * w);
#pragma unroll
          for (int u = 0; u < kQ4TPW; ++u) kw[u] = ldsm_x4(kc_base + u * kTile + okl);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int G = 2 * w + e;
            const uint4 qh = lds128a(qf_addr + G * 1024);
            const uint4 ql = lds128a(qf_addr + G * 1024 + 512);
#pragma unroll
            for (int u = 0; u < kQ4TPW; ++u) {
              const uint4 A = tq4_levels8(e ? kw[u].z : kw[u].x);  // key g: elements 8t .. 8t+7
              const uint4 B = tq4_levels8(e ? kw[u].w : kw[u].y);  // key g + 8
              float (&part)[4] = S[u][0];
              mma_f16(part, A.x, B.x, A.y, B.y, qh.x, qh.y);
              mma_f16(part, A.z, B.z, A.w, B.w, qh.z, qh.w);
              mma_f16(part, A.x, B.x, A.y, B.y, ql.x, ql.y);
              mma_f16(part, A.z, B.z, A.w, B.w, ql.z, ql.w);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kQ4TPW; ++u) {
          const uint32_t sb = ks_base + u * kQ4ScaleBytes;
          const float sa = lds16h(sb + 2 * g), sc = lds16h(sb + 2 * (g + 8));
          S[u][0][0] *= sa;
          S[u][0][1] *= sa;
          S[u][0][2] *= sc;
          S[u][0][3] *= sc;
        }
      } else {
        q4_score_tiles<GATHER, NT, kQ4TPW>(S, kc_base, ks_base, qf_addr, qb_addr, lrow, lhi, lane);
      }
      // (Dead columns have a zero query: their scores are 0, finite, and never
      // leave the kernel, so they need no mask.)
#pragma unroll
      for (int u = 0; u < kQ4TPW; ++u) {
        const int kt = k0 + 16 * (tile0 + u);  // the tile's first key
        if constexpr (WIN) {
          if (kt + 16 > Tmin) {  // warp-uniform: some row ends before the tile does
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                if (kt + g >= colen[nt][cc]) S[u][nt][cc] = -INFINITY;
                if (kt + g + 8 >= colen[nt][cc]) S[u][nt][2 + cc] = -INFINITY;
              }
          }
        } else {
          const int nvalid = k1 - kt;
          if (nvalid < 16) {  // warp-uniform: keys past the end (or a tile past the partition)
            if (g >= nvalid) S[u][0][0] = S[u][0][1] = -INFINITY;
            if (g + 8 >= nvalid) S[u][0][2] = S[u][0][3] = -INFINITY;
          }
        }
      }

      // The K tiles are consumed: refill them with round r + 1.
      __syncwarp();
      if (r + 1 < nrounds)
        poisoned |= q4_issue_own<GATHER, TQ, kQ4TPW>(a, b, kvh, k0, k1, r + 1, warp, lane, tile_row, grow, &a.tm_k, c.k,
                                                     c.k_scale, sm.kc[warp], sm.ks[warp], &sm.kbar[warp]);
    }

    // ---------------- round maximum, shared through shared memory
    float t0[NT], t1[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      t0[nt] = fmaxf(S[0][nt][0], S[0][nt][2]);
      t1[nt] = fmaxf(S[0][nt][1], S[0][nt][3]);
#pragma unroll
      for (int u = 1; u < kQ4TPW; ++u) {
        t0[nt] = fmaxf(t0[nt], fmaxf(S[u][nt][0], S[u][nt][2]));
        t1[nt] = fmaxf(t1[nt], fmaxf(S[u][nt][1], S[u][nt][3]));
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        t0[nt] = fmaxf(t0[nt], __shfl_xor_sync(0xffffffffu, t0[nt], o));
        t1[nt] = fmaxf(t1[nt], __shfl_xor_sync(0xffffffffu, t1[nt], o));
      }
      if (g == 0) *reinterpret_cast<float2*>(&sm.red[warp][8 * nt + 2 * t]) = make_float2(t0[nt], t1[nt]);
    }
    bar_sync_cta();  // (1) maxima published; every warp is past the P.V of round r - 1
    if constexpr (VR == 2) {
      // slot (r + 1) % 2 held round r - 1's V, which every warp is done with: round r + 1's
      if (r >= 1 && r + 1 < nrounds)
        poisoned |= q4_issue_own<GATHER, TQ, kQ4TPW>(a, b, kvh, k0, k1, r + 1, warp, lane, tile_row, grow, &a.tm_v, c.v, c.v_scale,
                                         &sm.vc[(r + 1) & 1][kQ4TPW * warp], &sm.vs[(r + 1) & 1][kQ4TPW * warp],
                                         &sm.vfull[(r + 1) & 1]);
    }
    {
      const uint32_t ra = smem_u32(&sm.red[0][2 * t]);
#pragma unroll
      for (int w = 0; w < kQ4Warps; ++w)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float2 mx = lds64f(ra + w * (32 * NT) + 32 * nt);
          t0[nt] = fmaxf(t0[nt], mx.x);
          t1[nt] = fmaxf(t1[nt], mx.y);
        }
    }

    // ---------------- online softmax (base 2), identical in every warp
    // n is finite (m starts at kQ4NoMax); c is exactly 1 while a column's maximum stands
    float c0[NT], c1[NT];
    bool moved = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const float n0 = fmaxf(m0[nt], t0[nt]), n1 = fmaxf(m1[nt], t1[nt]);
      c0[nt] = fast_exp2(m0[nt] - n0);
      c1[nt] = fast_exp2(m1[nt] - n1);
      m0[nt] = n0;
      m1[nt] = n1;
#pragma unroll
      for (int u = 0; u < kQ4TPW; ++u) {
        z0[u][nt] *= c0[nt];
        z1[u][nt] *= c1[nt];
      }
      moved |= c0[nt] != 1.f || c1[nt] != 1.f;
    }
    if (r > 0 && __any_sync(0xffffffffu, moved)) {  // acc is still zero in round 0
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            acc[e][j][nt][0] *= c0[nt];
            acc[e][j][nt][1] *= c1[nt];
            acc[e][j][nt][2] *= c0[nt];
            acc[e][j][nt][3] *= c1[nt];
          }
    }
    // P (keys x columns) -> B fragments (keys on K, columns on N), published
#pragma unroll
    for (int u = 0; u < kQ4TPW; ++u)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float p0 = fast_exp2(S[u][nt][0] - m0[nt]), p1 = fast_exp2(S[u][nt][1] - m1[nt]);
        const float p2 = fast_exp2(S[u][nt][2] - m0[nt]), p3 = fast_exp2(S[u][nt][3] - m1[nt]);
        z0[u][nt] += p0 + p2;
        z1[u][nt] += p1 + p3;
        const uint32_t pb0 = movmatrix_trans(pack_half2(p0, p1));  // keys 2t, 2t+1 of column g
        const uint32_t pb1 = movmatrix_trans(pack_half2(p2, p3));  // keys 2t+8, 2t+9
        sm.pb[kQ4TPW * warp + u][nt][lane] = make_uint2(pb0, pb1);
      }
    bar_sync_cta();  // (2) every tile's P is published

    // ---------------- P.V over the round's tiles for groups 2w, 2w+1
    const int vslot = VR == 2 ? (r & 1) : 0;
    const uint32_t vpar = VR == 2 ? ((r >> 1) & 1) : par;
    if (!timed_out && !__all_sync(0xffffffffu, mbar_wait_bounded(&sm.vfull[vslot], vpar))) timed_out = true;
    const uint32_t vc_base = smem_u32(&sm.vc[0][0][0]) + vslot * kVcSlot;
    const uint32_t vs_base = smem_u32(&sm.vs[0][0][0]) + vslot * kVsSlot + 4 * warp;  // groups 2w, 2w + 1
    const uint32_t vs_tq = smem_u32(&sm.vs[0][0][0]) + vslot * kVsSlot;  // TQ4: one fp16 scale per key
    const bool tail_round = k0 + kQ4RoundTiles * 16 * (r + 1) > k1;  // CTA-uniform
    // Every tile of the round is visited.  Keys past the end (the tail of the
    // last tile, and the tiles the last round does not have) get zero V scales:
    // their P is zero too, and their codes, stale or not, are finite once
    // converted, so they add exactly nothing.  Only a tail round checks.
    auto pv_round = [&](auto tail_tag) {
      constexpr bool kTail = decltype(tail_tag)::value;
      if constexpr (TQ) {
#pragma unroll
        for (int j = 0; j < kQ4RoundTiles; ++j) {
          const uint2 pp = lds64a(pb_addr + j * 256);
          // V scales of keys (2t, 2t+1) and (2t+8, 2t+9), one per row
          const uint32_t sb = vs_tq + j * kQ4ScaleBytes;
          uint32_t slo = lds32a(sb + 4 * t), shi = lds32a(sb + 16 + 4 * t);
          if constexpr (kTail) {
            const int nvalid = k1 - (k0 + 16 * (kQ4RoundTiles * r + j));
            if (nvalid < 16) {  // CTA-uniform
              if (2 * t >= nvalid) slo &= 0xFFFF0000u;
              if (2 * t + 1 >= nvalid) slo &= 0x0000FFFFu;
              if (2 * t + 8 >= nvalid) shi &= 0xFFFF0000u;
              if (2 * t + 9 >= nvalid) shi &= 0x0000FFFFu;
            }
          }
          const uint32_t b0 = h2_as_u32(__hmul2(u32_as_h2(pp.x), u32_as_h2(slo)));
          const uint32_t b1 = h2_as_u32(__hmul2(u32_as_h2(pp.y), u32_as_h2(shi)));
          // words of keys g, g + 8 for groups 2w, 2w + 1; levels by key, then
          // transposed (movmatrix) to pairs of keys per value dim
          const uint4 vw = ldsm_x4(vc_base + j * kTile + off_vl);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const uint4 A = tq4_levels8(e ? vw.z : vw.x);  // key g, elements 8t .. 8t+7
            const uint4 B = tq4_levels8(e ? vw.w : vw.y);  // key g + 8
            // rows g / g + 8 of the first MMA: dims 8(g/2) + (g&1) + 0 / + 2; second: + 4 / + 6
            mma_f16(acc[e][0][0], movmatrix_trans(A.x), movmatrix_trans(A.y), movmatrix_trans(B.x),
                    movmatrix_trans(B.y), b0, b1);
            mma_f16(acc[e][1][0], movmatrix_trans(A.z), movmatrix_trans(A.w), movmatrix_trans(B.z),
                    movmatrix_trans(B.w), b0, b1);
          }
        }
      } else {
        q4_pv_tiles<kTail, GATHER, NT>(acc, pb_addr, vc_base, vs_base, off_vl, k0 + kQ4RoundTiles * 16 * r, k1,
                                          lane);
      }
    };
    if (tail_round)
      pv_round(std::true_type{});
    else
      pv_round(std::false_type{});

    // The round's V is consumed once every warp gets here: then each warp
    // refills its own V tiles with round r + 1 (a one-round ring).
    if constexpr (VR == 1) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.vempty);
      if (r + 1 < nrounds) {
        if (!timed_out && !__all_sync(0xffffffffu, mbar_wait_bounded(&sm.vempty, par))) timed_out = true;
        poisoned |= q4_issue_own<GATHER, TQ, kQ4TPW>(a, b, kvh, k0, k1, r + 1, warp, lane, tile_row, grow, &a.tm_v, c.v, c.v_scale,
                                         &sm.vc[0][kQ4TPW * warp], &sm.vs[0][kQ4TPW * warp], &sm.vfull[0]);
      }
    }
  }
  if (timed_out && lane == 0) set_status(a.status, KVQ_DEV_TIMEOUT);
  poisoned = __any_sync(0xffffffffu, poisoned || timed_out);

  // ---------------- reduce z across the 8 key-row lanes; sum over the tile slots
#pragma unroll
  for (int u = 0; u < kQ4TPW; ++u)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        z0[u][nt] += __shfl_xor_sync(0xffffffffu, z0[u][nt], o);
        z1[u][nt] += __shfl_xor_sync(0xffffffffu, z1[u][nt], o);
      }
      if (g == 0)
        *reinterpret_cast<float2*>(&sm.zs[kQ4TPW * warp + u][8 * nt + 2 * t]) = make_float2(z0[u][nt], z1[u][nt]);
    }
  if (poisoned && lane == 0) atomicOr(&sm.poison, 1);
  __syncthreads();
  const bool bad = sm.poison != 0;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    // columns 8 nt + 2t + cc: row b + row, head kvh * group + col - row * group;
    // a window row past its own end has no partial in this partition
    int64_t pi[2];
    bool live[2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int col = 8 * nt + 2 * t + cc, row = col / a.group;
      live[cc] = row < nr && (!WIN || k0 < colen[nt][cc]);
      pi[cc] = ((int64_t)(b + row) * a.Hq + kvh * a.group + col - row * a.group) * a.P + p;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      if constexpr (TQ) {
        // accumulator rows g, g + 8 of MMA j hold dims d0 + 4j + 0, + 2
        const int d0 = 32 * (2 * warp + e) + 8 * (g >> 1) + (g & 1);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          if (!live[cc]) continue;
          float* o = a.ws_acc + pi[cc] * kQ4D + d0;
          o[0] = bad ? NAN : acc[e][0][nt][cc];
          o[2] = bad ? NAN : acc[e][0][nt][2 + cc];
          o[4] = bad ? NAN : acc[e][1][nt][cc];
          o[6] = bad ? NAN : acc[e][1][nt][2 + cc];
        }
      } else {
        const int d = 32 * (2 * warp + e) + 4 * g;
        float4 o0 = make_float4(acc[e][0][nt][0], acc[e][1][nt][0], acc[e][0][nt][2], acc[e][1][nt][2]);
        float4 o1 = make_float4(acc[e][0][nt][1], acc[e][1][nt][1], acc[e][0][nt][3], acc[e][1][nt][3]);
        if (bad) o0 = o1 = make_float4(NAN, NAN, NAN, NAN);
        if (live[0]) *reinterpret_cast<float4*>(a.ws_acc + pi[0] * kQ4D + d) = o0;
        if (live[1]) *reinterpret_cast<float4*>(a.ws_acc + pi[1] * kQ4D + d) = o1;
      }
    }
    if (warp == 0 && g == 0) {
      float Z[2] = {0.f, 0.f};
#pragma unroll
      for (int u = 0; u < kQ4RoundTiles; ++u) {
        Z[0] += sm.zs[u][8 * nt + 2 * t];
        Z[1] += sm.zs[u][8 * nt + 2 * t + 1];
      }
      const float M[2] = {m0[nt], m1[nt]};
#pragma unroll
      for (int cc = 0; cc < 2; ++cc)
        if (live[cc]) {
          a.ws_m[pi[cc]] = bad ? NAN : M[cc];
          a.ws_z[pi[cc]] = bad ? NAN : Z[cc];
        }
    }
  }
  if constexpr (LM) {
    // every thread's partials are visible device-wide before the count
    __threadfence();
    __syncthreads();
    const int64_t grp = (int64_t)b * a.c.num_kv_heads + kvh;   // (sequence, KV head)
    const int blk = p / kMergeBlock, p0 = blk * kMergeBlock;
    const int nb = min(kMergeBlock, nparts - p0);             // partitions in this block
    const int nblk = (nparts + kMergeBlock - 1) / kMergeBlock;
    int32_t* bctr = a.merge_ctr + a.c.num_kv_heads * (int64_t)a.merge_B + grp * a.merge_nblk + blk;
    if (threadIdx.x == 0) sm.last = atomicAdd(bctr, 1) == nb - 1;
    __syncthreads();
    if (sm.last) {
      __threadfence();
      // the ring buffers are free now: weights [group][n], sums and maxima [group]
      float* wts = reinterpret_cast<float*>(&sm.kc[0][0][0]);
      const int64_t h0 = (int64_t)b * a.Hq + kvh * a.group;  // the group's first query head
      q4_fold(a.ws_m + h0 * a.P + p0, a.ws_z + h0 * a.P + p0, a.ws_acc + (h0 * a.P + p0) * kQ4D, a.P, nb, a.group,
              wts, &sm.red[0][0], false, a.merge_m + h0 * a.merge_nblk + blk, a.merge_z + h0 * a.merge_nblk + blk,
              a.merge_acc + (h0 * a.merge_nblk + blk) * kQ4D, a.merge_nblk, nullptr, false);
      if (threadIdx.x == 0) *bctr = 0;  // ready for the next launch
      __threadfence();
      __syncthreads();
      if (threadIdx.x == 0) sm.last = atomicAdd(a.merge_ctr + grp, 1) == nblk - 1;
      __syncthreads();
      if (sm.last) {
        __threadfence();
        q4_fold(a.merge_m + h0 * a.merge_nblk, a.merge_z + h0 * a.merge_nblk, a.merge_acc + h0 * a.merge_nblk * kQ4D,
                a.merge_nblk, nblk, a.group, wts, &sm.red[0][0], true, nullptr, nullptr, nullptr, 0,
                a.fused_out + h0 * kQ4D, a.q_rotate != 0);
        if (threadIdx.x == 0) a.merge_ctr[grp] = 0;
      }
    }
  }
  pdl_trigger();  // after this CTA's last write
}

template <bool GATHER, int NT, bool WIN, bool TQ = false, bool LM = false, int MINB = 0, int VR = 1>
cudaError_t launch_round(const DecodeArgs& a, dim3 grid, cudaStream_t s) {
  const size_t smem = sizeof(Q4Smem<NT, GATHER, VR>) + 1024;  // + slack for the 1024-byte alignment
  auto kern = decode_q4_round_kernel<GATHER, NT, WIN, TQ, LM, MINB, VR>;
  cudaError_t e = set_max_smem_once<decode_q4_round_kernel<GATHER, NT, WIN, TQ, LM, MINB, VR>>((int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, grid, dim3(kQ4Warps * 32), smem, s, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace q4r

// ---------------------------------------------------------------- warp-specialised form
// The same decode for grids that fit in one wave of two CTAs per SM (short
// contexts, where one CTA per SM sub-partition pair leaves the schedulers idle):
// 8 warps per CTA.  Warps 0-3 score and run the softmax as the round kernel's
// warps do (tiles 2w, 2w + 1 of each round); warps 4-7 run P.V as the round
// kernel's warps do (value groups 2w', 2w' + 1), one round behind.  The
// probabilities and rescale factors of round r pass through slot r mod 2 of a
// two-slot buffer, so the scores of round r + 1 overlap the P.V of round r.
// Every value is computed by the same code as in the round kernel, so the
// partials are the same bits.  Named barriers: 1 the scoring warps' maxima;
// 2 + s slot s published (scoring warps arrive, P.V warps wait); 4 + s slot s
// free again (the other way round); 6 the P.V warps are done with a round's V
// tiles.  Every warp runs every round, so each barrier is always completed.
namespace q4s {

using namespace q4r;
constexpr int kRoles = 4;  // warps per role

// kvq_decode_step's store of the new token (q4_store_new_token's work) by the 8
// warps: each warp's two (plane, group) pairs, with both pairs' value loads and
// the block-table load issued together rather than one after another.
__device__ __forceinline__ void q4s_store_new_token(const DecodeArgs& a, int b, int kvh, int32_t pos, int warp,
                                                    int lane) {
  constexpr int kTasks = 2 * kQ4NG / (2 * kRoles);
  const kvq_cache& c = a.c;
  const int64_t src = ((int64_t)b * c.num_kv_heads + kvh) * kQ4D + lane;
  float x[kTasks];
#pragma unroll
  for (int i = 0; i < kTasks; ++i) {
    const int task = warp + 2 * kRoles * i, plane = task >= kQ4NG ? 1 : 0, G = task - plane * kQ4NG;
    x[i] = load_act(plane ? a.new_v : a.new_k, a.new_dtype, src + 32 * G);
  }
  const int32_t page = a.block_tables[(int64_t)b * a.bt_stride + pos / c.page_size];
  if (page >= 0 && page < c.num_pages) {
    const int64_t row = ((int64_t)page * c.num_kv_heads + kvh) * c.page_size + pos % c.page_size;
    const bool rot = c.format == KVQ_FMT_Q4_HAD32;
#pragma unroll
    for (int i = 0; i < kTasks; ++i) {
      const int task = warp + 2 * kRoles * i, plane = task >= kQ4NG ? 1 : 0, G = task - plane * kQ4NG;
      __half s16;
      const uint32_t code = rot ? q4_group_code_warp<true>(x[i], lane, s16) : q4_group_code_warp<false>(x[i], lane, s16);
      q4_write_group_warp(static_cast<uint8_t*>(plane ? c.v : c.k) + row * (kQ4D / 2),
                          static_cast<uint16_t*>(plane ? c.v_scale : c.k_scale) + row * kQ4NG, G, code, s16, lane);
    }
    fence_proxy_async_global();
  }
  __syncthreads();
}
constexpr int kBarMax = 1, kBarFull = 2, kBarEmpty = 4, kBarPv = 6;

template <bool GATHER>
struct __align__(1024) SpecSmem {
  static constexpr int kTile = q4_tile_bytes<GATHER>();
  uint8_t kc[2][kRoles][2][kTile];      // K ring: round mod 2, scoring warp, its 2 tiles
  uint8_t vc[2][kQ4RoundTiles][kTile];  // V ring: round mod 2, tile
  uint16_t ks[2][kRoles][2][16 * 8];
  uint16_t vs[2][kQ4RoundTiles][16 * 8];
  uint4 qf[1][kQ4NG][2][32];
  float4 qb[1][kQ4NG][4];
  uint2 pb[2][kQ4RoundTiles][1][32];  // P of round r in slot r mod 2 (B fragments)
  float cf[2][8];                     // the round's rescale factor per column
  float red[2][kRoles][8];            // maxima: round mod 2, scoring warp, column
  float zs[kQ4RoundTiles][8];         // sums of the probabilities per tile slot
  uint64_t kbar[2][kRoles];
  uint64_t vfull[2];
  int poison;
  int32_t grow[GATHER ? kQ4GatherPart : 1];  // gather: the cache row of each of the partition's entries
};

__device__ __forceinline__ void nbar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void nbar_arrive(int id, int n) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// GATHER: the gather of selected positions (512-entry partitions, the rows
// resolved once per CTA into shared memory and copied by cp.async), otherwise
// the dense decode.
template <bool GATHER>
__global__ void __launch_bounds__(2 * kRoles * 32, 2) decode_q4_spec_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  SpecSmem<GATHER>& sm =
      *reinterpret_cast<SpecSmem<GATHER>*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int p = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const bool scorer = warp < kRoles;
  const int rw = warp & (kRoles - 1);  // the warp's index within its role

  // metadata before the wait on the previous kernel (as in the round kernel);
  // a gather's entries are checked against the sequence one by one instead
  const int32_t T = GATHER ? a.n_sel : a.seq_lens[b];
  const bool bad_len = !GATHER && (T < 0 || T > a.max_seq_len || (int64_t)T > (int64_t)a.max_pages * a.c.page_size);
  const int nparts = bad_len ? 0 : (T + a.part - 1) / a.part;
  const bool active = p < nparts;
  const int k0 = p * a.part;
  const int k1 = min(k0 + a.part, T);
  const int ntiles = active ? (k1 - k0 + 15) / 16 : 0;
  const int nrounds = (ntiles + kQ4RoundTiles - 1) / kQ4RoundTiles;
  int32_t tile_row = -1;
  bool bad_page = false;
  if (!GATHER && lane < ntiles) {
    const int key0 = k0 + 16 * lane;
    const int32_t page = a.block_tables[(int64_t)b * a.bt_stride + key0 / a.c.page_size];
    if (page < 0 || page >= a.c.num_pages)
      bad_page = true;
    else
      tile_row = static_cast<int32_t>(((int64_t)page * a.c.num_kv_heads + kvh) * a.c.page_size + key0 % a.c.page_size);
  }
  if (active && threadIdx.x == 0) {
    for (int k = 0; k < 2; ++k)
      for (int w = 0; w < kRoles; ++w) mbar_init(&sm.kbar[k][w], 2);
    for (int i = 0; i < 2; ++i) mbar_init(&sm.vfull[i], kQ4RoundTiles);
    sm.poison = 0;
    fence_barrier_init();
  }

  pdl_wait();
  if (bad_len) {
    if (threadIdx.x == 0 && p == 0 && kvh == 0) set_status(a.status, KVQ_DEV_BAD_LENGTH);
    return;  // the merge writes NaN for this sequence
  }
  if (!active) return;
  if (bad_page && warp == 0) set_status(a.status, KVQ_DEV_BAD_PAGE);
  __syncthreads();  // the mbarriers are initialised
  const int32_t* grow = nullptr;
  if constexpr (GATHER) {
    // the partition's selected rows, resolved once and in parallel (as the
    // round kernel's gather does)
    const int32_t Tseq = a.seq_lens[b];
    const int32_t* bt = a.block_tables + (int64_t)b * a.bt_stride;
    const int64_t tmax = (int64_t)a.max_pages * a.c.page_size;
    for (int i = threadIdx.x; i < k1 - k0; i += 2 * kRoles * 32) {
      const int32_t pos = a.sel[(int64_t)b * a.n_sel + k0 + i];
      int32_t row = -1;
      if (pos < 0 || pos >= Tseq || pos >= tmax) {
        set_status(a.status, KVQ_DEV_BAD_INDEX);
      } else {
        const int32_t pg = bt[pos / a.c.page_size];
        if (pg < 0 || pg >= a.c.num_pages)
          set_status(a.status, KVQ_DEV_BAD_PAGE);
        else
          row = static_cast<int32_t>(((int64_t)pg * a.c.num_kv_heads + kvh) * a.c.page_size + pos % a.c.page_size);
      }
      sm.grow[i] = row;
    }
    __syncthreads();
    grow = sm.grow;
  }

  const kvq_cache& c = a.c;
  bool poisoned = false;
  auto issue_k01 = [&]() {
    if (scorer) {
      poisoned = q4r::q4_issue_own<GATHER, false, 2>(a, b, kvh, k0, k1, 0, rw, lane, tile_row, grow, &a.tm_k, c.k,
                                                    c.k_scale, sm.kc[0][rw], sm.ks[0][rw], &sm.kbar[0][rw]);
      if (nrounds > 1)
        poisoned |= q4r::q4_issue_own<GATHER, false, 2>(a, b, kvh, k0, k1, 1, rw, lane, tile_row, grow, &a.tm_k, c.k,
                                                       c.k_scale, sm.kc[1][rw], sm.ks[1][rw], &sm.kbar[1][rw]);
    }
  };
  // the query loads go out ahead of the first rounds' copies (which would
  // otherwise queue before them); the fragments are built after the copies
  QueryLoads<2 * kRoles> qload;
  if (!GATHER && a.new_k != nullptr && p == (T - 1) / a.part) {
    // This CTA stores the new token first.  Rounds 0 and 1 do not hold it when
    // it lies at entry 256 or later of the partition: their K copies then go
    // out before the store (later rounds' copies are issued after it).
    const bool k01_first = T - 1 - k0 >= 2 * kQ4RoundTiles * 16;
    if (k01_first) issue_k01();
    q4s_store_new_token(a, b, kvh, T - 1, warp, lane);
    q4_query_load<2 * kRoles>(a, b, kvh, warp, lane, qload);
    if (!k01_first) issue_k01();
  } else {
    q4_query_load<2 * kRoles>(a, b, kvh, warp, lane, qload);
    issue_k01();
  }
  // V of rounds 0 and 1, after the query fragments: K(0), which the first
  // round waits for, goes out alone first
  auto issue_v01 = [&]() {
    poisoned = q4r::q4_issue_own<GATHER, false, 2>(a, b, kvh, k0, k1, 0, rw, lane, tile_row, grow, &a.tm_v, c.v, c.v_scale,
                                                  &sm.vc[0][2 * rw], &sm.vs[0][2 * rw], &sm.vfull[0]);
    if (nrounds > 1)
      poisoned |= q4r::q4_issue_own<GATHER, false, 2>(a, b, kvh, k0, k1, 1, rw, lane, tile_row, grow, &a.tm_v, c.v,
                                                     c.v_scale, &sm.vc[1][2 * rw], &sm.vs[1][2 * rw], &sm.vfull[1]);
  };
  q4_query_build<2 * kRoles>(a, warp, lane, qload, sm.qf[0], sm.qb[0]);
  if (!scorer) issue_v01();
  const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lhi = lane >> 4;
  bool timed_out = false;
  float m0 = kQ4NoMax, m1 = kQ4NoMax;
  float z0[2][1] = {{0.f}, {0.f}}, z1[2][1] = {{0.f}, {0.f}};
  float acc[2][2][1][4];
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[e][j][0][i] = 0.f;

  if (scorer) {
    // ---------------- scores and softmax of tiles 2 rw, 2 rw + 1 of every round
    const uint32_t qf_addr = smem_u32(&sm.qf[0][0][0][lane]);
    const uint32_t qb_addr = smem_u32(&sm.qb[0][0][t]);
    for (int r = 0; r < nrounds; ++r) {
      const int s = r & 1;
      const uint32_t kc_base = smem_u32(&sm.kc[s][rw][0][0]), ks_base = smem_u32(&sm.ks[s][rw][0][0]);
      const int tile0 = kQ4RoundTiles * r + 2 * rw;
      float S[2][1][4];
#pragma unroll
      for (int u = 0; u < 2; ++u) S[u][0][0] = S[u][0][1] = S[u][0][2] = S[u][0][3] = -INFINITY;
      if (k0 + 16 * tile0 < k1) {  // warp-uniform
        if (!timed_out && !__all_sync(0xffffffffu, mbar_wait_bounded(&sm.kbar[s][rw], (r >> 1) & 1))) timed_out = true;
#pragma unroll
        for (int u = 0; u < 2; ++u) S[u][0][0] = S[u][0][1] = S[u][0][2] = S[u][0][3] = 0.f;
        q4_score_tiles<GATHER, 1, 2>(S, kc_base, ks_base, qf_addr, qb_addr, lrow, lhi, lane);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int nvalid = k1 - (k0 + 16 * (tile0 + u));
          if (nvalid < 16) {  // warp-uniform
            if (g >= nvalid) S[u][0][0] = S[u][0][1] = -INFINITY;
            if (g + 8 >= nvalid) S[u][0][2] = S[u][0][3] = -INFINITY;
          }
        }
        __syncwarp();  // the K tiles are consumed: refill the slot with round r + 2
        if (r + 2 < nrounds)
          poisoned |= q4r::q4_issue_own<GATHER, false, 2>(a, b, kvh, k0, k1, r + 2, rw, lane, tile_row, grow, &a.tm_k, c.k,
                                                         c.k_scale, sm.kc[s][rw], sm.ks[s][rw], &sm.kbar[s][rw]);
      }
      // round maximum over the scoring warps
      float t0 = fmaxf(S[0][0][0], S[0][0][2]), t1 = fmaxf(S[0][0][1], S[0][0][3]);
      t0 = fmaxf(t0, fmaxf(S[1][0][0], S[1][0][2]));
      t1 = fmaxf(t1, fmaxf(S[1][0][1], S[1][0][3]));
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, o));
        t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, o));
      }
      if (g == 0) *reinterpret_cast<float2*>(&sm.red[s][rw][2 * t]) = make_float2(t0, t1);
      nbar_sync(kBarMax, kRoles * 32);
#pragma unroll
      for (int w = 0; w < kRoles; ++w) {
        const float2 mx = *reinterpret_cast<const float2*>(&sm.red[s][w][2 * t]);
        t0 = fmaxf(t0, mx.x);
        t1 = fmaxf(t1, mx.y);
      }
      // online softmax (base 2), as in the round kernel
      const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);
      const float c0 = fast_exp2(m0 - n0), c1 = fast_exp2(m1 - n1);
      m0 = n0;
      m1 = n1;
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        z0[u][0] *= c0;
        z1[u][0] *= c1;
      }
      if (r >= 2) nbar_sync(kBarEmpty + s, 2 * kRoles * 32);  // the P.V warps are done with slot s
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float p0 = fast_exp2(S[u][0][0] - m0), p1 = fast_exp2(S[u][0][1] - m1);
        const float p2 = fast_exp2(S[u][0][2] - m0), p3 = fast_exp2(S[u][0][3] - m1);
        z0[u][0] += p0 + p2;
        z1[u][0] += p1 + p3;
        const uint32_t pb0 = movmatrix_trans(pack_half2(p0, p1));  // keys 2t, 2t+1 of column g
        const uint32_t pb1 = movmatrix_trans(pack_half2(p2, p3));  // keys 2t+8, 2t+9
        sm.pb[s][2 * rw + u][0][lane] = make_uint2(pb0, pb1);
      }
      if (rw == 0 && g == 0) *reinterpret_cast<float2*>(&sm.cf[s][2 * t]) = make_float2(c0, c1);
      nbar_arrive(kBarFull + s, 2 * kRoles * 32);
    }
  } else {
    // ---------------- P.V of value groups 2 rw, 2 rw + 1, one round behind the scores
    const uint32_t off_vl = q4_chunk_off<GATHER>(lrow, lhi, lane, 2 * rw);
    for (int r = 0; r < nrounds; ++r) {
      const int s = r & 1;
      nbar_sync(kBarFull + s, 2 * kRoles * 32);
      const float2 cc = *reinterpret_cast<const float2*>(&sm.cf[s][2 * t]);
      const bool moved = cc.x != 1.f || cc.y != 1.f;
      if (r > 0 && __any_sync(0xffffffffu, moved)) {  // acc is still zero in round 0
#pragma unroll
        for (int e = 0; e < 2; ++e)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            acc[e][j][0][0] *= cc.x;
            acc[e][j][0][1] *= cc.y;
            acc[e][j][0][2] *= cc.x;
            acc[e][j][0][3] *= cc.y;
          }
      }
      if (!timed_out && !__all_sync(0xffffffffu, mbar_wait_bounded(&sm.vfull[s], (r >> 1) & 1))) timed_out = true;
      const uint32_t vc_base = smem_u32(&sm.vc[s][0][0]);
      const uint32_t vs_base = smem_u32(&sm.vs[s][0][0]) + 4 * rw;
      const uint32_t pb_addr = smem_u32(&sm.pb[s][0][0][lane]);
      if (k0 + kQ4RoundTiles * 16 * (r + 1) > k1)  // CTA-uniform: the tail round
        q4_pv_tiles<true, GATHER, 1>(acc, pb_addr, vc_base, vs_base, off_vl, k0 + kQ4RoundTiles * 16 * r, k1, lane);
      else
        q4_pv_tiles<false, GATHER, 1>(acc, pb_addr, vc_base, vs_base, off_vl, k0 + kQ4RoundTiles * 16 * r, k1, lane);
      if (r + 2 < nrounds) nbar_arrive(kBarEmpty + s, 2 * kRoles * 32);  // slot s may take round r + 2
      nbar_sync(kBarPv, kRoles * 32);  // every P.V warp is done with the round's V tiles
      if (r + 2 < nrounds)
        poisoned |= q4r::q4_issue_own<GATHER, false, 2>(a, b, kvh, k0, k1, r + 2, rw, lane, tile_row, grow, &a.tm_v, c.v,
                                                       c.v_scale, &sm.vc[s][2 * rw], &sm.vs[s][2 * rw], &sm.vfull[s]);
    }
  }
  if (timed_out && lane == 0) set_status(a.status, KVQ_DEV_TIMEOUT);
  poisoned = __any_sync(0xffffffffu, poisoned || timed_out);
  if (scorer) {  // z: across the 8 key-row lanes, then per tile slot
#pragma unroll
    for (int u = 0; u < 2; ++u) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        z0[u][0] += __shfl_xor_sync(0xffffffffu, z0[u][0], o);
        z1[u][0] += __shfl_xor_sync(0xffffffffu, z1[u][0], o);
      }
      if (g == 0) *reinterpret_cast<float2*>(&sm.zs[2 * rw + u][2 * t]) = make_float2(z0[u][0], z1[u][0]);
    }
  }
  if (poisoned && lane == 0) atomicOr(&sm.poison, 1);
  __syncthreads();
  const bool bad = sm.poison != 0;
  int64_t pi[2];
  bool live[2];
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int col = 2 * t + cc;
    live[cc] = col < a.group;
    pi[cc] = ((int64_t)b * a.Hq + kvh * a.group + col) * a.P + p;
  }
  if (!scorer) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int d = 32 * (2 * rw + e) + 4 * g;
      float4 o0 = make_float4(acc[e][0][0][0], acc[e][1][0][0], acc[e][0][0][2], acc[e][1][0][2]);
      float4 o1 = make_float4(acc[e][0][0][1], acc[e][1][0][1], acc[e][0][0][3], acc[e][1][0][3]);
      if (bad) o0 = o1 = make_float4(NAN, NAN, NAN, NAN);
      if (live[0]) *reinterpret_cast<float4*>(a.ws_acc + pi[0] * kQ4D + d) = o0;
      if (live[1]) *reinterpret_cast<float4*>(a.ws_acc + pi[1] * kQ4D + d) = o1;
    }
  } else if (warp == 0 && g == 0) {
    float Z[2] = {0.f, 0.f};
#pragma unroll
    for (int u = 0; u < kQ4RoundTiles; ++u) {
      Z[0] += sm.zs[u][2 * t];
      Z[1] += sm.zs[u][2 * t + 1];
    }
    const float M[2] = {m0, m1};
#pragma unroll
    for (int cc = 0; cc < 2; ++cc)
      if (live[cc]) {
        a.ws_m[pi[cc]] = bad ? NAN : M[cc];
        a.ws_z[pi[cc]] = bad ? NAN : Z[cc];
      }
  }
  pdl_trigger();  // after this CTA's last write
}

template <bool GATHER>
cudaError_t launch_spec(const DecodeArgs& a, dim3 grid, cudaStream_t s) {
  const size_t smem = sizeof(SpecSmem<GATHER>) + 1024;  // + slack for the 1024-byte alignment
  cudaError_t e = set_max_smem_once<decode_q4_spec_kernel<GATHER>>((int)smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(decode_q4_spec_kernel<GATHER>, grid, dim3(2 * kRoles * 32), smem, s, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace q4s

bool decode_q4_one_wave(int64_t ctas) { return ctas <= 2 * static_cast<int64_t>(device_sm_count()); }

cudaError_t launch_decode_q4(const DecodeArgs& a, int B, cudaStream_t s) {
  using namespace q4r;
  if (a.nrows <= 0) {
    const dim3 grid(a.P, a.c.num_kv_heads, B);
    if (a.tq) return a.sel ? cudaErrorInvalidValue : launch_round<false, 1, false, true>(a, grid, s);
    const int64_t ctas = (int64_t)grid.x * grid.y * grid.z;
    const bool small = decode_q4_one_wave(ctas);
    if (a.fused_out)
      return a.sel ? cudaErrorInvalidValue
                   : small ? launch_round<false, 1, false, false, true, 2, 2>(a, grid, s)
                           : launch_round<false, 1, false, false, true>(a, grid, s);
    if (a.sel) {  // the resolved rows of a partition live in shared memory
      if (a.part != kQ4GatherPart) return cudaErrorInvalidValue;
      return small ? q4s::launch_spec<true>(a, grid, s) : launch_round<true, 1, false>(a, grid, s);
    }
    if (small) return q4s::launch_spec<false>(a, grid, s);
    return launch_round<false, 1, false>(a, grid, s);
  }
  if (a.tq) return cudaErrorInvalidValue;
  // Decode window: the rows are cut into the fewest even slices whose
  // (row, head) columns fit kQ4MaxColTiles tiles of 8.
  const int rmax = 8 * kQ4MaxColTiles / a.group;  // >= 4 (group <= 8)
  const int nslices = (a.nrows + rmax - 1) / rmax;
  DecodeArgs w = a;
  w.rows_per_cta = (a.nrows + nslices - 1) / nslices;
  const int nt = (w.rows_per_cta * a.group + 7) / 8;
  const dim3 grid(a.P, a.c.num_kv_heads, (a.nrows + w.rows_per_cta - 1) / w.rows_per_cta);
  switch (nt) {
    case 1: return launch_round<false, 1, true>(w, grid, s);
    case 2: return launch_round<false, 2, true>(w, grid, s);
    case 3: return launch_round<false, 3, true>(w, grid, s);
    default: return launch_round<false, 4, true>(w, grid, s);
  }
}

}  // namespace kvq
