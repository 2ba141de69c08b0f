// decode_fp8.cu -- split-T absorbed-MLA decode over fp8 e4m3 latent rows, on
// the tensor cores (mma.m16n8k16, f16 operands, f32 accumulation).
//
// Follows "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant": the KV8 base
// commit (a token is a 512-value latent row Lc and a 64-value rope row Rc, each
// e4m3 with one f32 scale; the score is Lsc.(q_L.Lc) + Rsc.(q_R.Rc) with the
// row scale outside the dot, and the latent row is also the value) and the
// split-T commit ((H, P) partial online-softmax blocks (cl, m, z) over
// 512-token partitions, merged by log-sum-exp; the selected-row gather of up to
// 4096 absolute indices splits into the same partials).
//
// GB300 design.  One CTA per (block of 32 query heads, partition of 512 tokens,
// sequence): 8 MMA warps and one producer warp.  Tokens stream in tiles of 64
// through a 2-stage shared-memory ring.  Dense tiles arrive by 2-D TMA: the
// latent codes as four 128-byte column boxes of 16 rows with the 128-byte
// swizzle, the rope codes as one 64-byte box with the 64-byte swizzle, the
// scales by 1-D bulk copies.  Gathered tiles arrive row by row (1-D bulk copies
// into rows padded to 528 / 80 bytes; scales by plain loads).
//  * Scores: heads on M (two 16-head blocks), tokens on N, the 576 dims on K.
//    The codes convert exactly to f16 (cvt of two e4m3 at once); the query is
//    split into f16 high and low parts (~22 bits) and stays in shared memory
//    in a permuted dim order, so that each lane's four code bytes of a k-step
//    are one 32-bit load.  Latent and rope dot products accumulate separately
//    and take their row scales in fp32.
//  * Softmax: a warp holds 16 tokens of 16 heads; row maxima over the tile's 64
//    tokens meet in shared memory; base-2 online softmax with running m per
//    head, partial z per warp.
//  * Context: P' = f16(p * Lsc) (shared memory) times the exact latent codes;
//    warp w owns output dims 64w .. 64w+63 for all 32 heads (64 f32
//    accumulators per thread); each lane reads 8 contiguous code bytes of a
//    token and builds the B fragments of 8 n-blocks from them (dim of n-block
//    nb, column n = 64w + 8n + nb).
#include <cuda_fp8.h>

#include "kernels.cuh"

namespace kvq {

constexpr int kF8Heads = 32;     // query heads per CTA
constexpr int kF8Keys = 64;      // tokens per tile
constexpr int kF8L = 512;        // latent width
constexpr int kF8R = 64;         // rope width
constexpr int kF8W = kF8L + kF8R;
constexpr int kF8Warps = 8;      // MMA warps; warp 8 is the producer
constexpr int kF8QStride = kF8W * 2 + 16;     // bytes per head row of q_hi / q_lo (padded)
constexpr int kF8PStride = kF8Keys * 2 + 16;  // bytes per head row of P'
constexpr int kF8GatherL = kF8L + 16;         // padded latent row (gather layout)
constexpr int kF8GatherR = kF8R + 16;         // padded rope row (gather layout)

struct __align__(1024) F8Stage {
  // dense: [4 column boxes][64 rows][128 B], 128-byte swizzled; gather: [64 rows][528 B]
  uint8_t lc[kF8Keys * kF8GatherL];
  // dense: [64 rows][64 B], 64-byte swizzled; gather: [64 rows][80 B]
  uint8_t rc[kF8Keys * kF8GatherR];
  float lsc[kF8Keys];
  float rsc[kF8Keys];
};

struct F8Smem {
  F8Stage stage[2];
  uint8_t qhi[kF8Heads * kF8QStride];
  uint8_t qlo[kF8Heads * kF8QStride];
  uint8_t p[kF8Heads * kF8PStride];
  float red[4][kF8Heads];   // per token quarter: tile row maxima
  float corr[kF8Heads];     // per head: rescale factor of this tile
  float zred[4][kF8Heads];  // end: partial z per token quarter
  uint64_t full[2], empty[2];
  int poison;
  int abort;
};
static_assert(sizeof(F8Smem) + 1024 <= 232448, "fp8 decode shared memory");

__device__ __forceinline__ void f8_tma_2d(void* dst, const CUtensorMap* map, int x, int row, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(row), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t f8_lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 f8_lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// Two e4m3 codes (low byte first) -> exact f16 pair.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t two_bytes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes & 0xFFFFu), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Byte offset of (token row r, latent byte d) in a stage.
template <bool GATHER>
__device__ __forceinline__ uint32_t lc_off(int r, int d) {
  if (GATHER) return r * kF8GatherL + d;
  return (d >> 7) * (kF8Keys * 128) + r * 128 + ((((d >> 4) & 7) ^ (r & 7)) << 4) + (d & 15);
}
// Byte offset of (token row r, rope byte d) in a stage.
template <bool GATHER>
__device__ __forceinline__ uint32_t rc_off(int r, int d) {
  if (GATHER) return r * kF8GatherR + d;
  return r * 64 + ((((d >> 4) & 3) ^ ((r >> 1) & 3)) << 4) + (d & 15);
}

// Bounded wait; once any warp has given up, the others stop waiting (they run
// on without data, so that every named barrier is still met; the output is NaN).
__device__ __forceinline__ bool f8_wait(F8Smem& sm, uint64_t* bar, uint32_t parity) {
  if (*reinterpret_cast<volatile int*>(&sm.abort)) return false;
  const bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
  if (!ok && (threadIdx.x & 31) == 0) atomicExch(&sm.abort, 1);
  return ok;
}

__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kF8Warps * 32) : "memory");
}

template <bool GATHER>
__global__ void __launch_bounds__((kF8Warps + 1) * 32, 1) decode_fp8_kernel(const __grid_constant__ DecodeArgs a) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  F8Smem& sm = *reinterpret_cast<F8Smem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int hblk = blockIdx.x, p = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const kvq_cache& c = a.c;
  const int head0 = hblk * kF8Heads;

  int32_t T;
  if (GATHER) {
    T = a.n_sel;
  } else {
    T = a.seq_lens[b];
    if (T < 0 || T > a.max_seq_len || (int64_t)T > (int64_t)a.max_pages * c.page_size) {
      if (threadIdx.x == 0 && p == 0 && hblk == 0) set_status(a.status, KVQ_DEV_BAD_LENGTH);
      return;  // the merge writes NaN for this sequence
    }
  }
  const int nparts = (T + kPart - 1) / kPart;
  if (p >= nparts) return;
  const int k0 = p * kPart;
  const int k1 = min(k0 + kPart, T);
  const int ntiles = (k1 - k0 + kF8Keys - 1) / kF8Keys;

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sm.full[s], 32);
      mbar_init(&sm.empty[s], kF8Warps);
    }
    sm.poison = 0;
    sm.abort = 0;
    fence_barrier_init();
  }
  // ---- queries: scaled, split, stored in the permuted dim order.  Within the
  // 16 dims of k-step s, k = 2t + j holds dim 16s + 4t + j and k = 8 + 2t + j
  // holds dim 16s + 4t + 2 + j (t = 0..3, j = 0, 1).
  for (int i = threadIdx.x; i < kF8Heads * (kF8W / 2); i += blockDim.x) {
    const int h = i / (kF8W / 2), kp = i % (kF8W / 2);  // k pair index
    const int s = kp >> 3, kk = 2 * (kp & 7);          // k-step, first k of the pair
    const int tt = (kk & 7) >> 1, hi8 = kk >> 3;
    const int d = 16 * s + 4 * tt + 2 * hi8;
    float x0 = 0.f, x1 = 0.f;
    if (head0 + h < a.Hq) {
      const float* qrow = a.q + ((int64_t)b * a.Hq + head0 + h) * kF8W;
      x0 = qrow[d] * a.qscale;
      x1 = qrow[d + 1] * a.qscale;
    }
    uint32_t hi, lo;
    split_f16(x0, x1, hi, lo);
    *reinterpret_cast<uint32_t*>(sm.qhi + h * kF8QStride + 2 * (16 * s + kk)) = hi;
    *reinterpret_cast<uint32_t*>(sm.qlo + h * kF8QStride + 2 * (16 * s + kk)) = lo;
  }
  __syncthreads();

  if (warp == kF8Warps) {
    // ---------------- producer warp
    const int32_t* bt = a.block_tables + (int64_t)b * a.max_pages;
    const int32_t Tseq = GATHER ? a.seq_lens[b] : T;
    bool bad = false;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      if (j >= 2 && !f8_wait(sm, &sm.empty[s], ((j >> 1) - 1) & 1)) break;
      F8Stage& st = sm.stage[s];
      const int key0 = k0 + j * kF8Keys;
      const int nvalid = min(kF8Keys, k1 - key0);
      if (!GATHER) {
        // lanes 0..3: one 16-token page chunk each
        uint32_t bytes = 0;
        int64_t row0 = -1;
        if (lane < 4 && 16 * lane < nvalid) {
          const int kk = key0 + 16 * lane;
          const int32_t page = bt[kk / c.page_size];
          if (page < 0 || page >= c.num_pages) {
            set_status(a.status, KVQ_DEV_BAD_PAGE);
            bad = true;
          } else {
            row0 = (int64_t)page * c.page_size + kk % c.page_size;
            bytes = 4 * 16 * 128 + 16 * 64 + 2 * 16 * 4;
          }
        }
        mbar_arrive_expect_tx(&sm.full[s], bytes);
        if (row0 >= 0) {
          const int r = 16 * lane;
#pragma unroll
          for (int x = 0; x < 4; ++x)
            f8_tma_2d(st.lc + x * (kF8Keys * 128) + r * 128, &a.tm_k, 128 * x, static_cast<int>(row0), &sm.full[s]);
          f8_tma_2d(st.rc + r * 64, &a.tm_v, 0, static_cast<int>(row0), &sm.full[s]);
          bulk_g2s(st.lsc + r, static_cast<const float*>(c.k_scale) + row0, 64, &sm.full[s]);
          bulk_g2s(st.rsc + r, static_cast<const float*>(c.v_scale) + row0, 64, &sm.full[s]);
        }
      } else {
        // each lane: tokens lane and lane + 32 of the tile
        uint32_t bytes = 0;
        int64_t rows[2] = {-1, -1};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int r = lane + 32 * u;
          if (r >= nvalid) continue;
          const int32_t pos = a.sel[(int64_t)b * a.n_sel + key0 + r];
          int32_t page = -1;
          if (pos < 0 || pos >= Tseq) {
            set_status(a.status, KVQ_DEV_BAD_INDEX);
            bad = true;
            continue;
          }
          page = bt[pos / c.page_size];
          if (page < 0 || page >= c.num_pages) {
            set_status(a.status, KVQ_DEV_BAD_PAGE);
            bad = true;
            continue;
          }
          rows[u] = (int64_t)page * c.page_size + pos % c.page_size;
          bytes += kF8L + kF8R;
        }
        // scales by plain loads (4-byte rows are below the bulk-copy granule)
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int r = lane + 32 * u;
          st.lsc[r] = rows[u] >= 0 ? static_cast<const float*>(c.k_scale)[rows[u]] : 0.f;
          st.rsc[r] = rows[u] >= 0 ? static_cast<const float*>(c.v_scale)[rows[u]] : 0.f;
        }
        mbar_arrive_expect_tx(&sm.full[s], bytes);  // release orders the scale stores
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (rows[u] < 0) continue;
          const int r = lane + 32 * u;
          bulk_g2s(st.lc + r * kF8GatherL, static_cast<const uint8_t*>(c.k) + rows[u] * kF8L, kF8L, &sm.full[s]);
          bulk_g2s(st.rc + r * kF8GatherR, static_cast<const uint8_t*>(c.v) + rows[u] * kF8R, kF8R, &sm.full[s]);
        }
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&sm.poison, 1);
  } else {
    // ---------------- MMA warps
    const int mb = warp & 1;   // head block of the scores
    const int nq = warp >> 1;  // token quarter of the scores: tokens 16 nq .. 16 nq + 15
    const uint32_t qhi_a = smem_u32(sm.qhi), qlo_a = smem_u32(sm.qlo), p_a = smem_u32(sm.p);
    // ldmatrix row addresses: matrix lane / 8 (rows 0-7 / 8-15, k-chunk 0 / 1), row lane % 8
    const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lchunk = lane >> 4;
    const uint32_t q_lane = (mb * 16 + lrow) * kF8QStride + 16 * lchunk;
    float m_run[2] = {-INFINITY, -INFINITY};  // heads mb*16 + g, + 8
    float z_part[2] = {0.f, 0.f};
    float acc[2][8][4];  // [head block][n-block][C fragment]: dims 64 warp + 8 n + nb
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[x][n][i] = 0.f;

    for (int j = 0; j < ntiles; ++j) {
      const int s = j & 1;
      f8_wait(sm, &sm.full[s], (j >> 1) & 1);
      const F8Stage& st = sm.stage[s];
      const uint32_t lc_a = smem_u32(st.lc), rc_a = smem_u32(st.rc);
      const int key0 = k0 + j * kF8Keys;
      const int nvalid = min(kF8Keys, k1 - key0);

      // ---------------- scores for tokens 16 nq + 8 f + n, f = 0, 1
      float cl[2][2][4], cr[2][2][4];  // [f][hi/lo][C]
#pragma unroll
      for (int f = 0; f < 2; ++f)
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int i = 0; i < 4; ++i) cl[f][u][i] = cr[f][u][i] = 0.f;
      const int kr0 = 16 * nq + g, kr1 = kr0 + 8;  // the B-fragment token rows of this lane
#pragma unroll 4
      for (int ks = 0; ks < kF8L / 16; ++ks) {
        uint32_t ah0, ah1, ah2, ah3, al0, al1, al2, al3;
        ldsm_x4(qhi_a + q_lane + 32 * ks, ah0, ah1, ah2, ah3);
        ldsm_x4(qlo_a + q_lane + 32 * ks, al0, al1, al2, al3);
        const uint32_t w0 = f8_lds32(lc_a + lc_off<GATHER>(kr0, 16 * ks + 4 * t));
        const uint32_t w1 = f8_lds32(lc_a + lc_off<GATHER>(kr1, 16 * ks + 4 * t));
        const uint32_t b00 = e4m3x2_to_h2(w0), b01 = e4m3x2_to_h2(w0 >> 16);
        const uint32_t b10 = e4m3x2_to_h2(w1), b11 = e4m3x2_to_h2(w1 >> 16);
        mma_f16(cl[0][0], ah0, ah1, ah2, ah3, b00, b01);
        mma_f16(cl[0][1], al0, al1, al2, al3, b00, b01);
        mma_f16(cl[1][0], ah0, ah1, ah2, ah3, b10, b11);
        mma_f16(cl[1][1], al0, al1, al2, al3, b10, b11);
      }
#pragma unroll
      for (int ks = 0; ks < kF8R / 16; ++ks) {
        uint32_t ah0, ah1, ah2, ah3, al0, al1, al2, al3;
        ldsm_x4(qhi_a + q_lane + 32 * (kF8L / 16 + ks), ah0, ah1, ah2, ah3);
        ldsm_x4(qlo_a + q_lane + 32 * (kF8L / 16 + ks), al0, al1, al2, al3);
        const uint32_t w0 = f8_lds32(rc_a + rc_off<GATHER>(kr0, 16 * ks + 4 * t));
        const uint32_t w1 = f8_lds32(rc_a + rc_off<GATHER>(kr1, 16 * ks + 4 * t));
        const uint32_t b00 = e4m3x2_to_h2(w0), b01 = e4m3x2_to_h2(w0 >> 16);
        const uint32_t b10 = e4m3x2_to_h2(w1), b11 = e4m3x2_to_h2(w1 >> 16);
        mma_f16(cr[0][0], ah0, ah1, ah2, ah3, b00, b01);
        mma_f16(cr[0][1], al0, al1, al2, al3, b00, b01);
        mma_f16(cr[1][0], ah0, ah1, ah2, ah3, b10, b11);
        mma_f16(cr[1][1], al0, al1, al2, al3, b10, b11);
      }
      // C fragment of (f): rows (heads) g, g + 8; columns (tokens) 16 nq + 8 f + 2t, + 1
      float sc[2][4];
      float lsc[2][2];  // [f][token 2t, 2t+1]
#pragma unroll
      for (int f = 0; f < 2; ++f) {
        const int kc = 16 * nq + 8 * f + 2 * t;
        const float2 ls = *reinterpret_cast<const float2*>(&st.lsc[kc]);
        const float2 rs = *reinterpret_cast<const float2*>(&st.rsc[kc]);
        // rows past the end hold stale or unwritten bytes: their P' must be an exact 0
        lsc[f][0] = kc < nvalid ? ls.x : 0.f;
        lsc[f][1] = kc + 1 < nvalid ? ls.y : 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float l = cl[f][0][i] + cl[f][1][i], r = cr[f][0][i] + cr[f][1][i];
          const int kcol = kc + (i & 1);
          float v = fmaf((i & 1) ? ls.y : ls.x, l, ((i & 1) ? rs.y : rs.x) * r);
          if (kcol >= nvalid) v = -INFINITY;
          sc[f][i] = v;
        }
      }
      // row maxima over this warp's 16 tokens, then over the tile's 64
      float t0 = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));  // head g
      float t1 = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));  // head g + 8
      t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, 1));
      t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, 2));
      t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, 1));
      t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, 2));
      if (t == 0) {
        sm.red[nq][mb * 16 + g] = t0;
        sm.red[nq][mb * 16 + g + 8] = t1;
      }
      consumers_sync();
      float tm0 = -INFINITY, tm1 = -INFINITY;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        tm0 = fmaxf(tm0, sm.red[u][mb * 16 + g]);
        tm1 = fmaxf(tm1, sm.red[u][mb * 16 + g + 8]);
      }
      const float n0 = fmaxf(m_run[0], tm0), n1 = fmaxf(m_run[1], tm1);
      const float u0 = (n0 == -INFINITY) ? 0.f : n0, u1 = (n1 == -INFINITY) ? 0.f : n1;
      const float c0 = fast_exp2(m_run[0] - u0), c1 = fast_exp2(m_run[1] - u1);
      m_run[0] = n0;
      m_run[1] = n1;
      float zs0 = 0.f, zs1 = 0.f;
#pragma unroll
      for (int f = 0; f < 2; ++f) {
        const float p0 = fast_exp2(sc[f][0] - u0), p1 = fast_exp2(sc[f][1] - u0);
        const float p2 = fast_exp2(sc[f][2] - u1), p3 = fast_exp2(sc[f][3] - u1);
        zs0 += p0 + p1;
        zs1 += p2 + p3;
        const int kc = 16 * nq + 8 * f + 2 * t;
        *reinterpret_cast<uint32_t*>(sm.p + (mb * 16 + g) * kF8PStride + 2 * kc) =
            pack_half2(p0 * lsc[f][0], p1 * lsc[f][1]);
        *reinterpret_cast<uint32_t*>(sm.p + (mb * 16 + g + 8) * kF8PStride + 2 * kc) =
            pack_half2(p2 * lsc[f][0], p3 * lsc[f][1]);
      }
      z_part[0] = fmaf(z_part[0], c0, zs0);
      z_part[1] = fmaf(z_part[1], c1, zs1);
      if (nq == 0 && t == 0) {
        sm.corr[mb * 16 + g] = c0;
        sm.corr[mb * 16 + g + 8] = c1;
      }
      consumers_sync();

      // ---------------- context: O[32 heads][dims 64 warp ..] += P' . Lc
      {
        float cf[2][2];  // [head block][row g / g + 8]
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          cf[x][0] = sm.corr[x * 16 + g];
          cf[x][1] = sm.corr[x * 16 + g + 8];
        }
        if (j > 0 && __any_sync(0xffffffffu, cf[0][0] != 1.f || cf[0][1] != 1.f || cf[1][0] != 1.f ||
                                                  cf[1][1] != 1.f)) {
#pragma unroll
          for (int x = 0; x < 2; ++x)
#pragma unroll
            for (int n = 0; n < 8; ++n) {
              acc[x][n][0] *= cf[x][0];
              acc[x][n][1] *= cf[x][0];
              acc[x][n][2] *= cf[x][1];
              acc[x][n][3] *= cf[x][1];
            }
        }
      }
      const int dbase = 64 * warp + 8 * g;  // this lane's 8 latent bytes of a token
#pragma unroll
      for (int ks = 0; ks < kF8Keys / 16; ++ks) {
        uint32_t a0[4], a1[4];
        ldsm_x4(p_a + (0 * 16 + lrow) * kF8PStride + 16 * (2 * ks + lchunk), a0[0], a0[1], a0[2], a0[3]);
        ldsm_x4(p_a + (1 * 16 + lrow) * kF8PStride + 16 * (2 * ks + lchunk), a1[0], a1[1], a1[2], a1[3]);
        const int r0 = 16 * ks + 2 * t;
        uint2 v0 = f8_lds64(lc_a + lc_off<GATHER>(r0, dbase));
        uint2 v1 = f8_lds64(lc_a + lc_off<GATHER>(r0 + 1, dbase));
        uint2 v2 = f8_lds64(lc_a + lc_off<GATHER>(r0 + 8, dbase));
        uint2 v3 = f8_lds64(lc_a + lc_off<GATHER>(r0 + 9, dbase));
        if (nvalid < kF8Keys) {  // tail tile: stale code bytes (possibly NaN codes) must not meet P' = 0
          if (r0 >= nvalid) v0 = make_uint2(0, 0);
          if (r0 + 1 >= nvalid) v1 = make_uint2(0, 0);
          if (r0 + 8 >= nvalid) v2 = make_uint2(0, 0);
          if (r0 + 9 >= nvalid) v3 = make_uint2(0, 0);
        }
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
          const uint32_t sel = (nb & 3) | ((4 + (nb & 3)) << 4);
          const uint32_t lo = (nb < 4) ? prmt(v0.x, v1.x, sel) : prmt(v0.y, v1.y, sel);
          const uint32_t hi = (nb < 4) ? prmt(v2.x, v3.x, sel) : prmt(v2.y, v3.y, sel);
          const uint32_t b0 = e4m3x2_to_h2(lo), b1 = e4m3x2_to_h2(hi);
          mma_f16(acc[0][nb], a0[0], a0[1], a0[2], a0[3], b0, b1);
          mma_f16(acc[1][nb], a1[0], a1[1], a1[2], a1[3], b0, b1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty[s]);
    }

    pdl_trigger();
    // ---------------- partials
    z_part[0] += __shfl_xor_sync(0xffffffffu, z_part[0], 1);
    z_part[0] += __shfl_xor_sync(0xffffffffu, z_part[0], 2);
    z_part[1] += __shfl_xor_sync(0xffffffffu, z_part[1], 1);
    z_part[1] += __shfl_xor_sync(0xffffffffu, z_part[1], 2);
    if (t == 0) {
      sm.zred[nq][mb * 16 + g] = z_part[0];
      sm.zred[nq][mb * 16 + g + 8] = z_part[1];
    }
    consumers_sync();
    const bool bad = sm.poison != 0 || sm.abort != 0;
    if (sm.abort != 0 && threadIdx.x == 0) set_status(a.status, KVQ_DEV_TIMEOUT);
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int hl = x * 16 + g + 8 * hr;
        if (head0 + hl >= a.Hq) continue;
        const int64_t pi = ((int64_t)b * a.Hq + head0 + hl) * a.P + p;
        float* dst = a.ws_acc + pi * kF8L;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb) {
          // columns n = 2t, 2t + 1 of n-block nb: dims 64 warp + 8n + nb
          dst[64 * warp + 8 * (2 * t) + nb] = bad ? NAN : acc[x][nb][2 * hr];
          dst[64 * warp + 8 * (2 * t + 1) + nb] = bad ? NAN : acc[x][nb][2 * hr + 1];
        }
        if (warp < 2 && t == 0 && x == mb) {
          // the m of a head is the same in the four warps of its block
          a.ws_m[pi] = bad ? NAN : m_run[hr];
          a.ws_z[pi] = bad ? NAN : sm.zred[0][hl] + sm.zred[1][hl] + sm.zred[2][hl] + sm.zred[3][hl];
        }
      }
  }
}

cudaError_t launch_decode_fp8(const DecodeArgs& a, int B, cudaStream_t s) {
  const size_t smem = sizeof(F8Smem) + 1024;
  const dim3 grid((a.Hq + kF8Heads - 1) / kF8Heads, a.P, B);
  if (a.sel) {
    cudaError_t e =
        cudaFuncSetAttribute(decode_fp8_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_fp8_kernel<true>, grid, dim3((kF8Warps + 1) * 32), smem, s, a);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e =
        cudaFuncSetAttribute(decode_fp8_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_fp8_kernel<false>, grid, dim3((kF8Warps + 1) * 32), smem, s, a);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace kvq
