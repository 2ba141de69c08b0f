// decode_q4.cu -- split-T decode attention over the Hadamard-rotated 4-bit cache.
//
// Follows "qwen27 CUDA: an opt-in 4-bit attention cache (262K on a 24 GB card)",
// section "What it is": attend over the 4-bit cache in rotated space, in shared
// 512-key chunks plus the tail, producing per-chunk partials that are merged in
// order; and "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", split-T
// commit: (H, P) partial online-softmax blocks (cl, m, z) + a log-sum-exp merge.
//
// GB300 design.  One CTA (4 warps) per (partition of 512 keys, KV head,
// sequence); up to 3 CTAs per SM.  Warp w owns keys [128w, 128w + 128) of the
// partition: 8 tiles of 16 keys streamed through a private 2-stage shared-memory
// ring.  A tile is 2 KB of K codes and 2 KB of V codes, brought by 2-D TMA
// tensor copies with the hardware 128-byte swizzle (16-byte chunk c of row r
// lands at chunk c ^ (r & 7), so the fragment loads below are free of bank
// conflicts), plus 256 B of K scales and 256 B of V scales by 1-D bulk copies.
// Fragment words are read one group pair at a time, so that few registers stay
// live besides the 64 output accumulators.  (Measured at 262K keys: the loads
// alone would run in ~56 us and the arithmetic alone in ~82 us; the kernel is
// bound by its arithmetic issue, not by the copies.)
//  * Scores on the tensor cores: mma.m16n8k16, the 16 keys on M, the <= 8 query
//    heads of the GQA group on N.  The key codes enter as the exact f16 values
//    1024 + c / 1024 + 16c (one lop3 per pair); the constant part is removed by
//    starting each group's accumulator at a per-(head, group) query bias.  The
//    query is split into f16 high and low parts (~22 bits; its fragments sit in
//    shared memory); each 32-value group gets its own partial product multiplied
//    by the group's fp32 scale, so the dequantised keys enter exactly.
//  * Online softmax in base 2 (the query carries sm_scale * log2 e).
//  * P.V on the tensor cores with the value dims on M: the probabilities are
//    transposed in registers (movmatrix) and multiplied by the V group scale in
//    f16; V codes minus 8 are exact in f16.
// The four warps' (m, z, acc) are combined in shared memory into the
// partition's partial.  The gather variant (selected rows) copies row by row
// with 1-D bulk copies into an unswizzled ring.
#include "kernels.cuh"

namespace kvq {

constexpr int kQ4Warps = 4;      // warps per CTA; each owns kPart / kQ4Warps keys of the partition
constexpr int kQ4MinBlocks = 3;  // resident CTAs per SM the register budget is sized for
constexpr int kQ4Ring = 2;       // tiles in flight per warp
constexpr int kQ4TilesPerWarp = kPart / 16 / kQ4Warps;  // 8
constexpr int kQ4D = 256;
constexpr int kQ4NG = 8;

// Stage layout (1024-byte aligned for the 128-byte swizzle of the code tiles).
struct __align__(1024) Q4Stage {
  uint8_t kc[16 * 128];  // K codes, swizzled (dense) or plain (gather)
  uint8_t vc[16 * 128];  // V codes
  uint16_t ks[16 * 8];   // K scales
  uint16_t vs[16 * 8];   // V scales
  uint8_t pad[512];
};
static_assert(sizeof(Q4Stage) == 5120, "stage size");

struct Q4Smem {
  Q4Stage stage[kQ4Warps][kQ4Ring];
  uint4 qf[kQ4NG][2][32];  // query fragments [group][hi, lo][lane]
  float2 qbias[kQ4NG][4];  // [group][head pair]: the code offset folded into the score MMA
  float qrot[8][kQ4D];     // the group's queries rotated in the kernel (unrotated-query entry point)
  uint64_t bar[kQ4Warps][kQ4Ring];
  int poison;
};

struct Q4Combine {  // reuses the ring once every warp is done
  float acc[kQ4Warps][8][kQ4D];
  float m[kQ4Warps][8];
  float z[kQ4Warps][8];
};
static_assert(sizeof(Q4Combine) <= sizeof(Q4Stage) * kQ4Warps * kQ4Ring, "combine fits in the ring");

__device__ __forceinline__ void tma_rows_2d(void* dst, const CUtensorMap* map, int row, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(smem_u32(bar))
      : "memory");
}

// Issue the copies of one 16-key tile into `st`.  Returns false if a page or a
// selected index is invalid (the tile then counts as poisoned; its barrier is
// still completed so the consumer does not wait on it).
template <bool GATHER>
__device__ __forceinline__ bool q4_issue_tile(const DecodeArgs& a, int b, int kvh, int key0, int nvalid,
                                              int32_t page, Q4Stage* st, uint64_t* bar) {
  const kvq_cache& c = a.c;
  const int32_t* bt = a.block_tables + (int64_t)b * a.max_pages;
  if constexpr (!GATHER) {
    // `page` is the block-table entry of key0, fetched ahead by the caller
    if (page < 0 || page >= c.num_pages) {
      set_status(a.status, KVQ_DEV_BAD_PAGE);
      mbar_arrive(bar);
      return false;
    }
    const int64_t row0 = ((int64_t)page * c.num_kv_heads + kvh) * c.page_size + key0 % c.page_size;
    mbar_arrive_expect_tx(bar, 2 * 16 * 128 + 2 * 16 * 16);
    tma_rows_2d(st->kc, &a.tm_k, static_cast<int>(row0), bar);
    tma_rows_2d(st->vc, &a.tm_v, static_cast<int>(row0), bar);
    bulk_g2s(st->ks, static_cast<const uint16_t*>(c.k_scale) + row0 * 8, 16 * 16, bar);
    bulk_g2s(st->vs, static_cast<const uint16_t*>(c.v_scale) + row0 * 8, 16 * 16, bar);
    return true;
  } else {
    const int32_t T = a.seq_lens[b];
    int64_t rows[16];
    for (int j = 0; j < nvalid; ++j) {
      const int32_t pos = a.sel[(int64_t)b * a.n_sel + key0 + j];
      int32_t page = -1;
      if (pos < 0 || pos >= T) {
        set_status(a.status, KVQ_DEV_BAD_INDEX);
      } else {
        page = bt[pos / c.page_size];
        if (page < 0 || page >= c.num_pages) set_status(a.status, KVQ_DEV_BAD_PAGE);
      }
      if (page < 0 || page >= c.num_pages) {
        mbar_arrive(bar);
        return false;
      }
      rows[j] = ((int64_t)page * c.num_kv_heads + kvh) * c.page_size + pos % c.page_size;
    }
    mbar_arrive_expect_tx(bar, nvalid * 288);
    for (int j = 0; j < nvalid; ++j) {
      bulk_g2s(st->kc + j * 128, static_cast<const uint8_t*>(c.k) + rows[j] * 128, 128, bar);
      bulk_g2s(st->vc + j * 128, static_cast<const uint8_t*>(c.v) + rows[j] * 128, 128, bar);
      bulk_g2s(st->ks + j * 8, static_cast<const uint16_t*>(c.k_scale) + rows[j] * 8, 16, bar);
      bulk_g2s(st->vs + j * 8, static_cast<const uint16_t*>(c.v_scale) + rows[j] * 8, 16, bar);
    }
    return true;
  }
}

// shared-memory loads at a 32-bit shared address
__device__ __forceinline__ uint4 lds128a(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
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

__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ float scale_of(const uint4& v, int G) {
  const uint32_t w = word_of(v, G >> 1);
  return __half2float(__ushort_as_half(static_cast<uint16_t>((G & 1) ? (w >> 16) : (w & 0xFFFFu))));
}

template <bool GATHER>
__global__ void __launch_bounds__(kQ4Warps * 32, kQ4MinBlocks) decode_q4_kernel(const __grid_constant__ DecodeArgs a) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled tiles (the launch adds 1 KB of slack)
  Q4Smem& sm = *reinterpret_cast<Q4Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int p = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;

  int32_t T;
  if (GATHER) {
    T = a.n_sel;
  } else {
    T = a.seq_lens[b];
    if (T < 0 || T > a.max_seq_len || (int64_t)T > (int64_t)a.max_pages * a.c.page_size) {
      if (threadIdx.x == 0 && p == 0 && kvh == 0) set_status(a.status, KVQ_DEV_BAD_LENGTH);
      return;  // the merge writes NaN for this sequence
    }
  }
  const int nparts = (T + kPart - 1) / kPart;
  if (p >= nparts) return;
  const int k0 = p * kPart;
  const int k1 = min(k0 + kPart, T);
  const int ntiles = (k1 - k0 + 15) / 16;
  const int my_first = warp * kQ4TilesPerWarp;
  const int my_tiles = max(0, min(kQ4TilesPerWarp, ntiles - my_first));

  // Page id of each of this warp's tiles, one per lane, fetched once (the
  // producer lane then never waits on a global load inside the tile loop).
  int32_t my_page = -1;
  if (!GATHER && lane < my_tiles)
    my_page = a.block_tables[(int64_t)b * a.max_pages + (k0 + 16 * (my_first + lane)) / a.c.page_size];
  int32_t first_pages[kQ4Ring];
#pragma unroll
  for (int i = 0; i < kQ4Ring; ++i) first_pages[i] = __shfl_sync(0xffffffffu, my_page, i);

  bool poisoned = false;
  if (lane == 0) {
    for (int s = 0; s < kQ4Ring; ++s) mbar_init(&sm.bar[warp][s], 1);
    fence_barrier_init();
    for (int i = 0; i < min(kQ4Ring, my_tiles); ++i) {
      const int key0 = k0 + 16 * (my_first + i);
      if (!q4_issue_tile<GATHER>(a, b, kvh, key0, min(16, k1 - key0), first_pages[i], &sm.stage[warp][i],
                                 &sm.bar[warp][i]))
        poisoned = true;
    }
  }
  if (threadIdx.x == 0) sm.poison = 0;

  // ---- query fragments (B operand of the score MMA), written once by warp 0.
  // The K codes enter the MMA as 1024 + c (even elements, low nibbles) and
  // 1024 + 16c (odd elements, high nibbles), one lop3 each; the query values
  // facing high nibbles are pre-divided by 16 (exact), and the accumulator of
  // group G starts at -bias_G, bias_G = 1024 * sum(B) + 8 * sum(q~) over the
  // group (B the f16 values in the fragments, q~ = B or 16 B), so the MMA
  // returns sum_d q_d (c_d - 8) with the keys' codes used exactly.
  const float* qsrc = a.q + ((int64_t)b * a.Hq + kvh * a.group) * kQ4D;  // rows of the group's heads
  if (a.q_raw) {
    // Rotate the group's queries here, with the arithmetic of the rotation entry
    // point (fp32 butterfly, stages 1..16, one multiply by fp32(1/sqrt(32))):
    // warp w takes (head, group) pairs w, w + 4, ..., lane = element.
    // All loads first (at most 8 heads x 8 groups / 4 warps = 16 per lane), so
    // their latencies overlap; then the butterflies.
    constexpr int kPairs = 8 * kQ4NG / kQ4Warps;
    const int npairs = a.group * kQ4NG;
    const int64_t qbase = ((int64_t)b * a.Hq + kvh * a.group) * kQ4D + lane;
    float xs[kPairs];
#pragma unroll
    for (int k = 0; k < kPairs; ++k) {
      const int hg = warp + kQ4Warps * k;  // (head, group) = (hg / 8, hg % 8): elements 32 hg .. of the rows
      xs[k] = 0.f;
      if (hg < npairs)
        xs[k] = a.q_dtype == KVQ_DT_F32
                    ? static_cast<const float*>(a.q_raw)[qbase + 32 * hg]
                    : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q_raw)[qbase + 32 * hg]);
    }
#pragma unroll
    for (int k = 0; k < kPairs; ++k) {
      const int hg = warp + kQ4Warps * k;
      if (hg < npairs) {  // warp-uniform
        const float x = warp_fwht32(xs[k], lane);
        (&sm.qrot[0][0])[32 * hg + lane] = __fmul_rn(x, kHadamardScale);
      }
    }
    __syncthreads();
    qsrc = &sm.qrot[0][0];
  }
  {
    const bool live = g < a.group;
    const float* qrow = qsrc + (live ? g : 0) * kQ4D;
    const float s = live ? a.qscale : 0.f;
    const float s16 = s * 0.0625f;
    constexpr int kGroupsPerWarp = kQ4NG / kQ4Warps;
    float4 ql0[kGroupsPerWarp], ql1[kGroupsPerWarp];  // all loads issued first
#pragma unroll
    for (int k = 0; k < kGroupsPerWarp; ++k) {
      ql0[k] = *reinterpret_cast<const float4*>(qrow + 32 * (warp + kQ4Warps * k) + 8 * t);
      ql1[k] = *reinterpret_cast<const float4*>(qrow + 32 * (warp + kQ4Warps * k) + 8 * t + 4);
    }
#pragma unroll
    for (int k = 0; k < kGroupsPerWarp; ++k) {  // warp w prepares groups w, w + kQ4Warps, ...
      const int G = warp + kQ4Warps * k;
      const float4 u0 = ql0[k];
      const float4 u1 = ql1[k];
      uint4 hi, lo;
      // tile (G,0): slots (2t,2t+1) <- d (8t, 8t+2); slots (2t+8, 2t+9) <- d (8t+1, 8t+3); tile (G,1): d + 4
      split_f16(u0.x * s, u0.z * s, hi.x, lo.x);
      split_f16(u0.y * s16, u0.w * s16, hi.y, lo.y);
      split_f16(u1.x * s, u1.z * s, hi.z, lo.z);
      split_f16(u1.y * s16, u1.w * s16, hi.w, lo.w);
      sm.qf[G][0][lane] = hi;
      sm.qf[G][1][lane] = lo;
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
      // bias = 1024 (ev + od) + 8 (ev + 16 od), summed over the 4 lanes of the head
      float bias = 1032.f * ev + 1152.f * od;
      bias += __shfl_xor_sync(0xffffffffu, bias, 1);
      bias += __shfl_xor_sync(0xffffffffu, bias, 2);
      // head g's bias -> qbias[G][g/2].x or .y
      if (t == 0) reinterpret_cast<float*>(&sm.qbias[G][0])[g] = -bias;
    }
  }
  __syncthreads();
  const uint32_t qf_addr = smem_u32(&sm.qf[0][0][lane]);
  const uint32_t qb_addr = smem_u32(&sm.qbias[0][t]);

  float acc[kQ4NG][2][4];
#pragma unroll
  for (int G = 0; G < kQ4NG; ++G)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[G][e][i] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;  // running max of heads 2t, 2t+1 (base 2)
  float z0 = 0.f, z1 = 0.f;              // this thread's partial sums
  const bool head0_live = 2 * t < a.group, head1_live = 2 * t + 1 < a.group;
  bool timed_out = false;

  // Byte offsets of this thread's fragments inside a stage (swizzle: chunk ^ (row & 7)).
  const int sw = GATHER ? 0 : g;       // rows g and g+8 share (row & 7) = g
  const int swv = GATHER ? 0 : 2 * t;  // rows 2t, 2t+8 -> 2t ; rows 2t+1, 2t+9 -> 2t+1
  const uint32_t off_ka0 = g * 128 + (((2 * t) ^ sw) << 4);
  const uint32_t off_ka1 = g * 128 + (((2 * t + 1) ^ sw) << 4);
  const uint32_t off_kb0 = off_ka0 + 8 * 128;
  const uint32_t off_kb1 = off_ka1 + 8 * 128;
  const uint32_t off_v0 = 2048 + (2 * t) * 128 + ((g ^ swv) << 4);
  const uint32_t off_v1 = 2048 + (2 * t + 1) * 128 + ((g ^ (GATHER ? 0 : swv + 1)) << 4);
  const uint32_t off_v2 = off_v0 + 8 * 128;
  const uint32_t off_v3 = off_v1 + 8 * 128;

  for (int i = 0; i < my_tiles; ++i) {
    const int s = i % kQ4Ring;
    Q4Stage& st = sm.stage[warp][s];
    // mma.sync / movmatrix below are warp-collective: the wait's outcome is made
    // warp-uniform so that the warp stays converged (also when a wait gives up).
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sm.bar[warp][s], (i / kQ4Ring) & 1))) {
      timed_out = true;
      break;
    }
    const uint32_t sbase = smem_u32(&st);
    const int key0 = k0 + 16 * (my_first + i);
    const int nvalid = min(16, k1 - key0);

    // ---------------- scores S[key][head] for keys g, g+8 and heads 2t, 2t+1
    float S[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kQ4NG / 2; ++w) {  // group pair (2w, 2w+1): one word of each fragment row
      const uint32_t wa0 = lds32a(sbase + off_ka0 + 4 * w);  // half-words (2t, G = 2w, 2w+1) of row g
      const uint32_t wa1 = lds32a(sbase + off_ka1 + 4 * w);  // half-words (2t+1, G)
      const uint32_t wb0 = lds32a(sbase + off_kb0 + 4 * w);  // row g+8
      const uint32_t wb1 = lds32a(sbase + off_kb1 + 4 * w);
      const __half2 sca = u32_as_h2(lds32a(sbase + 4096 + g * 16 + 4 * w));  // K scales (2w, 2w+1) of row g
      const __half2 scb = u32_as_h2(lds32a(sbase + 4096 + (g + 8) * 16 + 4 * w));
      const float2 fsa = __half22float2(sca), fsb = __half22float2(scb);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int G = 2 * w + e;
        const uint4 qh = lds128a(qf_addr + G * 1024);
        const uint4 ql = lds128a(qf_addr + G * 1024 + 512);
        const uint2 nb = lds64a(qb_addr + G * 32);  // -bias of heads 2t, 2t+1
        const uint32_t sel = e ? 0x4342u : 0x4140u;
        const uint32_t xa1 = prmt(wa0, 0u, sel);
        const uint32_t xa2 = prmt(wa1, 0u, sel);
        const uint32_t xb1 = prmt(wb0, 0u, sel);
        const uint32_t xb2 = prmt(wb1, 0u, sel);
        const uint32_t a10 = nib_lo_pair_biased(xa1), a11 = nib_lo_pair_biased(xb1);
        const uint32_t a12 = nib_hi_pair_biased(xa1), a13 = nib_hi_pair_biased(xb1);
        const uint32_t a20 = nib_lo_pair_biased(xa2), a21 = nib_lo_pair_biased(xb2);
        const uint32_t a22 = nib_hi_pair_biased(xa2), a23 = nib_hi_pair_biased(xb2);
        float part[4] = {__uint_as_float(nb.x), __uint_as_float(nb.y), __uint_as_float(nb.x), __uint_as_float(nb.y)};
        mma_f16(part, a10, a11, a12, a13, qh.x, qh.y);
        mma_f16(part, a20, a21, a22, a23, qh.z, qh.w);
        mma_f16(part, a10, a11, a12, a13, ql.x, ql.y);
        mma_f16(part, a20, a21, a22, a23, ql.z, ql.w);
        const float sa = e ? fsa.y : fsa.x, sb = e ? fsb.y : fsb.x;
        S[0] = fmaf(sa, part[0], S[0]);
        S[1] = fmaf(sa, part[1], S[1]);
        S[2] = fmaf(sb, part[2], S[2]);
        S[3] = fmaf(sb, part[3], S[3]);
      }
    }
    if (!head0_live) S[0] = S[2] = -INFINITY;
    if (!head1_live) S[1] = S[3] = -INFINITY;
    if (nvalid < 16) {  // tail tile: mask keys past the end
      if (g >= nvalid) S[0] = S[1] = -INFINITY;
      if (g + 8 >= nvalid) S[2] = S[3] = -INFINITY;
    }

    // ---------------- online softmax (base 2)
    float t0 = fmaxf(S[0], S[2]), t1 = fmaxf(S[1], S[3]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, o));
      t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, o));
    }
    const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);
    const float u0 = (n0 == -INFINITY) ? 0.f : n0, u1 = (n1 == -INFINITY) ? 0.f : n1;
    const float c0 = fast_exp2(m0 - u0), c1 = fast_exp2(m1 - u1);
    const float p0 = fast_exp2(S[0] - u0), p1 = fast_exp2(S[1] - u1);
    const float p2 = fast_exp2(S[2] - u0), p3 = fast_exp2(S[3] - u1);
    z0 = fmaf(z0, c0, p0 + p2);
    z1 = fmaf(z1, c1, p1 + p3);
    m0 = n0;
    m1 = n1;
    if (i > 0 && __any_sync(0xffffffffu, c0 != 1.f || c1 != 1.f)) {  // acc is still zero on the first tile
#pragma unroll
      for (int G = 0; G < kQ4NG; ++G)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          acc[G][e][0] *= c0;
          acc[G][e][1] *= c1;
          acc[G][e][2] *= c0;
          acc[G][e][3] *= c1;
        }
    }

    // ---------------- P (keys x heads) -> B fragments (keys on K, heads on N)
    const uint32_t pb0 = movmatrix_trans(pack_half2(p0, p1));  // keys 2t, 2t+1 of head g
    const uint32_t pb1 = movmatrix_trans(pack_half2(p2, p3));  // keys 2t+8, 2t+9

    // V scales of keys 2t, 2t+1, 2t+8, 2t+9 (zero past the end) and V codes of
    // the same rows (half-word h = g of every group), loaded one group pair at a
    // time so that few registers stay live.
    const bool va_ok = 2 * t < nvalid, vb_ok = 2 * t + 1 < nvalid;
    const bool vc_ok = 2 * t + 8 < nvalid, vd_ok = 2 * t + 9 < nvalid;
#pragma unroll
    for (int w = 0; w < kQ4NG / 2; ++w) {
      const uint32_t swa = va_ok ? lds32a(sbase + 4352 + (2 * t) * 16 + 4 * w) : 0u;
      const uint32_t swb = vb_ok ? lds32a(sbase + 4352 + (2 * t + 1) * 16 + 4 * w) : 0u;
      const uint32_t swc = vc_ok ? lds32a(sbase + 4352 + (2 * t + 8) * 16 + 4 * w) : 0u;
      const uint32_t swd = vd_ok ? lds32a(sbase + 4352 + (2 * t + 9) * 16 + 4 * w) : 0u;
      const uint32_t cw0 = lds32a(sbase + off_v0 + 4 * w);
      const uint32_t cw1 = lds32a(sbase + off_v1 + 4 * w);
      const uint32_t cw2 = lds32a(sbase + off_v2 + 4 * w);
      const uint32_t cw3 = lds32a(sbase + off_v3 + 4 * w);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int G = 2 * w + e;
        const uint32_t ssel = e ? 0x7632u : 0x5410u;
        const uint32_t slo = prmt(swa, swb, ssel);
        const uint32_t shi = prmt(swc, swd, ssel);
        const uint32_t b0 = h2_as_u32(__hmul2(u32_as_h2(pb0), u32_as_h2(slo)));
        const uint32_t b1 = h2_as_u32(__hmul2(u32_as_h2(pb1), u32_as_h2(shi)));
        const uint32_t s0 = e ? 0x6622u : 0x4400u;  // byte X of rows a, b -> bytes 0, 2
        const uint32_t s1 = e ? 0x7733u : 0x5511u;  // byte X+1
        const uint32_t x01 = prmt(cw0, cw1, s0);
        const uint32_t x01b = prmt(cw0, cw1, s1);
        const uint32_t x23 = prmt(cw2, cw3, s0);
        const uint32_t x23b = prmt(cw2, cw3, s1);
        // d-tile (G,0): rows g <-> d = 32G+4g, g+8 <-> 32G+4g+2 ; (G,1): +1
        mma_f16(acc[G][0], nib_lo_pair(x01), nib_lo_pair(x01b), nib_lo_pair(x23), nib_lo_pair(x23b), b0, b1);
        mma_f16(acc[G][1], nib_hi_pair(x01), nib_hi_pair(x01b), nib_hi_pair(x23), nib_hi_pair(x23b), b0, b1);
      }
    }

    const int32_t next_page = __shfl_sync(0xffffffffu, my_page, min(i + kQ4Ring, 31));
    __syncwarp();
    if (lane == 0 && i + kQ4Ring < my_tiles) {
      fence_proxy_async();
      const int nk0 = k0 + 16 * (my_first + i + kQ4Ring);
      if (!q4_issue_tile<GATHER>(a, b, kvh, nk0, min(16, k1 - nk0), next_page, &st, &sm.bar[warp][s]))
        poisoned = true;
    }
  }
  if (timed_out && lane == 0) set_status(a.status, KVQ_DEV_TIMEOUT);
  poisoned = __any_sync(0xffffffffu, poisoned || timed_out);

  // ---------------- reduce z across the 8 key-row lanes
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    z0 += __shfl_xor_sync(0xffffffffu, z0, o);
    z1 += __shfl_xor_sync(0xffffffffu, z1, o);
  }
  if (poisoned && lane == 0) atomicOr(&sm.poison, 1);
  __syncthreads();  // every warp is done with the ring
  Q4Combine& cb = *reinterpret_cast<Q4Combine*>(&sm.stage[0][0]);
#pragma unroll
  for (int G = 0; G < kQ4NG; ++G) {
    const int d = 32 * G + 4 * g;
    *reinterpret_cast<float4*>(&cb.acc[warp][2 * t][d]) =
        make_float4(acc[G][0][0], acc[G][1][0], acc[G][0][2], acc[G][1][2]);
    *reinterpret_cast<float4*>(&cb.acc[warp][2 * t + 1][d]) =
        make_float4(acc[G][0][1], acc[G][1][1], acc[G][0][3], acc[G][1][3]);
  }
  if (g == 0) {
    cb.m[warp][2 * t] = m0;
    cb.m[warp][2 * t + 1] = m1;
    cb.z[warp][2 * t] = z0;
    cb.z[warp][2 * t + 1] = z1;
  }
  __syncthreads();
  const bool bad = sm.poison != 0;
  for (int idx = threadIdx.x; idx < a.group * (kQ4D / 4); idx += blockDim.x) {
    const int h = idx / (kQ4D / 4), d4 = idx % (kQ4D / 4);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kQ4Warps; ++w) M = fmaxf(M, cb.m[w][h]);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float Z = 0.f;
#pragma unroll
    for (int w = 0; w < kQ4Warps; ++w) {
      const float wt = (M == -INFINITY) ? 0.f : exp2f(cb.m[w][h] - M);
      const float4 v = *reinterpret_cast<const float4*>(&cb.acc[w][h][4 * d4]);
      o.x = fmaf(v.x, wt, o.x);
      o.y = fmaf(v.y, wt, o.y);
      o.z = fmaf(v.z, wt, o.z);
      o.w = fmaf(v.w, wt, o.w);
      Z = fmaf(cb.z[w][h], wt, Z);
    }
    const int64_t pi = ((int64_t)b * a.Hq + kvh * a.group + h) * a.P + p;
    if (bad) o = make_float4(NAN, NAN, NAN, NAN);
    *reinterpret_cast<float4*>(a.ws_acc + pi * kQ4D + 4 * d4) = o;
    if (d4 == 0) {
      a.ws_m[pi] = bad ? NAN : M;
      a.ws_z[pi] = bad ? NAN : Z;
    }
  }
  pdl_trigger();  // after this CTA's last write
}

cudaError_t launch_decode_q4(const DecodeArgs& a, int B, cudaStream_t s) {
  const size_t smem = sizeof(Q4Smem) + 1024;
  dim3 grid(a.P, a.c.num_kv_heads, B);
  if (a.sel) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_q4_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_q4_kernel<true>, grid, dim3(kQ4Warps * 32), smem, s, a);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e =
        cudaFuncSetAttribute(decode_q4_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_q4_kernel<false>, grid, dim3(kQ4Warps * 32), smem, s, a);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace kvq
