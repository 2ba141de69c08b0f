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
// sequence): 8 MMA warps and one producer warp.  Tokens arrive in tiles of 64
// into one raw stage: dense tiles by 2-D TMA (the latent codes as four 128-byte
// column boxes of 16 rows with the 128-byte swizzle, the rope codes as one
// 64-byte box with the 64-byte swizzle, the scales by 1-D bulk copies);
// gathered tiles row by row (the latent rows by 1-D bulk copies, the rope rows
// and the scales by cp.async through the load path, into rows padded to 528 /
// 80 bytes), while the MMA warps split the query.
//  * The 8 MMA warps convert the tile once into an f16 tile in shared memory
//    (cvt of two e4m3 at once, exact; rows past the end become zeros), which
//    frees the raw stage for the next tile's copy while the MMAs run.
//  * Scores: heads on M (two 16-head blocks), tokens on N, the 576 dims on K;
//    A = the query split into f16 high and low parts (~22 bits) by ldmatrix,
//    B = the f16 tile by ldmatrix.  Latent and rope dot products accumulate
//    separately and take their row scales in fp32.
//  * Softmax: a warp holds 16 tokens of 16 heads; row maxima over the tile's 64
//    tokens meet in shared memory; base-2 online softmax with running m per
//    head, partial z per warp.
//  * Context: P' = f16(p * Lsc) (shared memory, A by ldmatrix) times the exact
//    latent values (B by ldmatrix.trans from the same f16 tile); warp w owns
//    output dims 64w .. 64w+63 for all 32 heads (64 f32 accumulators per thread).
// The prefill of a prompt chunk (the split-T commit's "tiled streaming kernel
// ... with the cap lifted to 1M") is this kernel with a whole row as its one
// partition: one CTA per (32 heads, row) streams every key of the row through
// the same tile loop, rows sharing one block table with lengths q_start + row + 1.
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
constexpr int kF8TStride = kF8W * 2 + 16;     // bytes per token row of the f16 tile (padded)

struct __align__(1024) F8Stage {
  // dense: [4 column boxes][64 rows][128 B], 128-byte swizzled; gather: [64 rows][528 B]
  uint8_t lc[kF8Keys * kF8GatherL];
  // dense: [64 rows][64 B], 64-byte swizzled; gather: [64 rows][80 B]
  uint8_t rc[kF8Keys * kF8GatherR];
  float lsc[kF8Keys];
  float rsc[kF8Keys];
};

struct F8Smem {
  F8Stage raw;
  uint8_t kf[kF8Keys * kF8TStride];  // the tile as f16: [token][576 values], natural order
  uint8_t qhi[kF8Heads * kF8QStride];
  uint8_t qlo[kF8Heads * kF8QStride];
  uint8_t p[kF8Heads * kF8PStride];
  float red[4][kF8Heads];   // per token quarter: tile row maxima
  float corr[kF8Heads];     // per head: rescale factor of this tile
  float zred[4][kF8Heads];  // end: partial z per token quarter
  uint64_t full, empty;
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

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint4 f8_lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
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
    T = a.prefill ? a.prefill_q0 + b + 1 : a.seq_lens[b];
    if (T < 0 || T > a.max_seq_len || (int64_t)T > (int64_t)a.max_pages * c.page_size) {
      if (threadIdx.x == 0 && p == 0 && hblk == 0) set_status(a.status, KVQ_DEV_BAD_LENGTH);
      return;  // the merge writes NaN for this sequence
    }
  }
  // partitions of a.part keys (512; a whole row for the streaming prefill)
  const int nparts = static_cast<int>(((int64_t)T + a.part - 1) / a.part);
  if (p >= nparts) return;
  const int k0 = p * a.part;
  const int k1 = static_cast<int>(min((int64_t)k0 + a.part, (int64_t)T));
  const int ntiles = (k1 - k0 + kF8Keys - 1) / kF8Keys;

  if (threadIdx.x == 0) {
    mbar_init(&sm.full, 32);         // the producer's lanes
    mbar_init(&sm.empty, kF8Warps);  // the MMA warps, once the raw tile is converted
    sm.poison = 0;
    sm.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();  // the barriers are initialised: the producer starts its copies at once
  // ---- queries: scaled by sm_scale * log2(e), split into f16 high and low parts
  // by the MMA warps while the producer's first tile is on its way (its row
  // indices are a chain of dependent loads when gathering).  32 heads x 144
  // float4 = 18 per thread; all loads are issued before any use.  The barrier
  // the MMA warps pass after the first tile lands orders these writes before
  // any score reads them.
  if (warp < kF8Warps) {
    constexpr int kUnits = kF8Heads * (kF8W / 4);
    constexpr int kPer = (kUnits + kF8Warps * 32 - 1) / (kF8Warps * 32);
    float4 v[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * kF8Warps * 32;
      const int h = i / (kF8W / 4), u = i % (kF8W / 4);
      v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < kUnits && head0 + h < a.Hq)
        v[k] = *reinterpret_cast<const float4*>(a.q + ((int64_t)b * a.Hq + head0 + h) * kF8W + 4 * u);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int i = threadIdx.x + k * kF8Warps * 32;
      if (i >= kUnits) break;
      const int h = i / (kF8W / 4), u = i % (kF8W / 4);
      uint2 hi, lo;
      split_f16(v[k].x * a.qscale, v[k].y * a.qscale, hi.x, lo.x);
      split_f16(v[k].z * a.qscale, v[k].w * a.qscale, hi.y, lo.y);
      *reinterpret_cast<uint2*>(sm.qhi + h * kF8QStride + 8 * u) = hi;
      *reinterpret_cast<uint2*>(sm.qlo + h * kF8QStride + 8 * u) = lo;
    }
  }

  if (warp == kF8Warps) {
    // ---------------- producer warp
    const int32_t* bt = a.block_tables + (int64_t)b * a.bt_stride;  // bt_stride 0: one table for every row
    const int32_t Tseq = GATHER ? a.seq_lens[b] : T;
    bool bad = false;
    F8Stage& st = sm.raw;
    for (int j = 0; j < ntiles; ++j) {
      if (j >= 1 && !f8_wait(sm, &sm.empty, (j - 1) & 1)) break;  // tile j - 1 converted
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
        mbar_arrive_expect_tx(&sm.full, bytes);
        if (row0 >= 0) {
          const int r = 16 * lane;
#pragma unroll
          for (int x = 0; x < 4; ++x)
            f8_tma_2d(st.lc + x * (kF8Keys * 128) + r * 128, &a.tm_k, 128 * x, static_cast<int>(row0), &sm.full);
          f8_tma_2d(st.rc + r * 64, &a.tm_v, 0, static_cast<int>(row0), &sm.full);
          bulk_g2s(st.lsc + r, static_cast<const float*>(c.k_scale) + row0, 64, &sm.full);
          bulk_g2s(st.rsc + r, static_cast<const float*>(c.v_scale) + row0, 64, &sm.full);
        }
      } else {
        // each lane: tokens lane and lane + 32 of the tile, resolved together
        // (both selected positions loaded, then both pages: two dependent
        // loads in all, not two per token)
        uint32_t bytes = 0;
        int64_t rows[2] = {-1, -1};
        int32_t pos[2], page[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int r = lane + 32 * u;
          pos[u] = r < nvalid ? a.sel[(int64_t)b * a.n_sel + key0 + r] : -1;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const bool in = lane + 32 * u < nvalid && pos[u] >= 0 && pos[u] < Tseq;
          page[u] = in ? bt[pos[u] / c.page_size] : -1;
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int r = lane + 32 * u;
          if (r >= nvalid) continue;
          if (pos[u] < 0 || pos[u] >= Tseq) {
            set_status(a.status, KVQ_DEV_BAD_INDEX);
            bad = true;
            continue;
          }
          if (page[u] < 0 || page[u] >= c.num_pages) {
            set_status(a.status, KVQ_DEV_BAD_PAGE);
            bad = true;
            continue;
          }
          rows[u] = (int64_t)page[u] * c.page_size + pos[u] % c.page_size;
          bytes += kF8L;
        }
        // The latent rows by bulk copies (their bytes expected before they are
        // issued), each lane's own two; the rope rows (4 x 16 bytes) and the
        // scales (4 bytes, below the bulk-copy granule; zeros for a row without
        // one) through the load path, so that the copy engine, which takes a
        // tile's copies one after another, queues only the 64 latent rows.  The
        // lane's arrival comes once its load-path copies have landed; the phase
        // also waits for the latent bytes.
        mbar_expect_tx(&sm.full, bytes);
        __syncwarp();  // every lane's bytes are expected before any copy can complete
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (rows[u] < 0) continue;
          const int r = lane + 32 * u;
          bulk_g2s(st.lc + r * kF8GatherL, static_cast<const uint8_t*>(c.k) + rows[u] * kF8L, kF8L, &sm.full);
        }
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int r = lane + 32 * u;
          const int64_t row = rows[u] >= 0 ? rows[u] : 0;
          if (rows[u] >= 0) {
#pragma unroll
            for (int x = 0; x < kF8R / 16; ++x)
              cp_async_16(st.rc + r * kF8GatherR + 16 * x, static_cast<const uint8_t*>(c.v) + row * kF8R + 16 * x);
          }
          const uint32_t n = rows[u] >= 0 ? 4u : 0u;
          cp_async_4(&st.lsc[r], static_cast<const float*>(c.k_scale) + row, n);
          cp_async_4(&st.rsc[r], static_cast<const float*>(c.v_scale) + row, n);
        }
        cp_async_mbar_arrive(&sm.full);
      }
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(&sm.poison, 1);
  } else {
    // ---------------- MMA warps
    const int mb = warp & 1;   // head block of the scores
    const int nq = warp >> 1;  // token quarter of the scores: tokens 16 nq .. 16 nq + 15
    const uint32_t qhi_a = smem_u32(sm.qhi), qlo_a = smem_u32(sm.qlo), p_a = smem_u32(sm.p);
    const uint32_t kf_a = smem_u32(sm.kf);
    const uint32_t lc_a = smem_u32(sm.raw.lc), rc_a = smem_u32(sm.raw.rc);
    // ldmatrix row addresses.  A (queries, P'): matrix lane / 8 = (rows 0-7 / 8-15) x
    // (k-chunk 0 / 1).  B of the scores (tile rows = tokens): (tokens 0-7, chunk 0),
    // (0-7, chunk 1), (8-15, chunk 0), (8-15, chunk 1).  B of the context (.trans):
    // (tokens 0-7, dims +0), (8-15, +0), (0-7, +8), (8-15, +8).
    const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1), lchunk = lane >> 4;
    const uint32_t q_lane = (mb * 16 + lrow) * kF8QStride + 16 * lchunk;
    const uint32_t ks_lane = kf_a + (16 * nq + (lane & 7) + 8 * (lane >> 4)) * kF8TStride + 16 * ((lane >> 3) & 1);
    const uint32_t kv_lane = kf_a + ((lane & 7) + 8 * ((lane >> 3) & 1)) * kF8TStride + 16 * (8 * warp + (lane >> 4));
    float m_run[2] = {-INFINITY, -INFINITY};  // heads mb*16 + g, + 8
    float z_part[2] = {0.f, 0.f};
    float acc[2][8][4];  // [head block][n-block][C fragment]: dims 64 warp + 8 nb + 2t, + 1
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[x][n][i] = 0.f;

    for (int j = 0; j < ntiles; ++j) {
      f8_wait(sm, &sm.full, j & 1);
      const int key0 = k0 + j * kF8Keys;
      const int nvalid = min(kF8Keys, k1 - key0);
      consumers_sync();  // every warp is done with the previous tile's f16 values

      // ---------------- convert the raw tile to f16 (rows past the end: zeros)
      static_assert(kF8Keys * (kF8W / 16) % (kF8Warps * 32) == 0, "conversion chunks per thread");
#pragma unroll
      for (int k = 0; k < kF8Keys * (kF8W / 16) / (kF8Warps * 32); ++k) {
        const int idx = threadIdx.x + k * (kF8Warps * 32);
        const int r = idx / (kF8W / 16), cchunk = idx % (kF8W / 16);  // 16 codes
        uint4 w = make_uint4(0, 0, 0, 0);
        if (r < nvalid)
          w = f8_lds128(cchunk < kF8L / 16 ? lc_a + lc_off<GATHER>(r, 16 * cchunk)
                                           : rc_a + rc_off<GATHER>(r, 16 * (cchunk - kF8L / 16)));
        const uint4 h0 = make_uint4(e4m3x2_to_h2(w.x), e4m3x2_to_h2(w.x >> 16), e4m3x2_to_h2(w.y),
                                    e4m3x2_to_h2(w.y >> 16));
        const uint4 h1 = make_uint4(e4m3x2_to_h2(w.z), e4m3x2_to_h2(w.z >> 16), e4m3x2_to_h2(w.w),
                                    e4m3x2_to_h2(w.w >> 16));
        uint8_t* dst = sm.kf + r * kF8TStride + 32 * cchunk;
        *reinterpret_cast<uint4*>(dst) = h0;
        *reinterpret_cast<uint4*>(dst + 16) = h1;
      }
      // the scales of this warp's score columns, read before the raw stage is released
      float ls[2][2], rs[2][2];  // [f][token 2t, 2t + 1]
#pragma unroll
      for (int f = 0; f < 2; ++f) {
        const int kc = 16 * nq + 8 * f + 2 * t;
        const float2 l2 = *reinterpret_cast<const float2*>(&sm.raw.lsc[kc]);
        const float2 r2 = *reinterpret_cast<const float2*>(&sm.raw.rsc[kc]);
        // rows past the end hold stale or unwritten bytes: their P' must be an exact 0
        ls[f][0] = kc < nvalid ? l2.x : 0.f;
        ls[f][1] = kc + 1 < nvalid ? l2.y : 0.f;
        rs[f][0] = kc < nvalid ? r2.x : 0.f;
        rs[f][1] = kc + 1 < nvalid ? r2.y : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.empty);  // the raw stage may be refilled
      consumers_sync();                       // the f16 tile is complete

      // ---------------- scores for tokens 16 nq + 8 f + n, f = 0, 1
      float cl[2][2][4], cr[2][2][4];  // [f][hi/lo][C]
#pragma unroll
      for (int f = 0; f < 2; ++f)
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int i = 0; i < 4; ++i) cl[f][u][i] = cr[f][u][i] = 0.f;
#pragma unroll 4
      for (int ks = 0; ks < kF8L / 16; ++ks) {
        uint32_t ah0, ah1, ah2, ah3, al0, al1, al2, al3, b00, b01, b10, b11;
        ldsm_x4(qhi_a + q_lane + 32 * ks, ah0, ah1, ah2, ah3);
        ldsm_x4(qlo_a + q_lane + 32 * ks, al0, al1, al2, al3);
        ldsm_x4(ks_lane + 32 * ks, b00, b01, b10, b11);
        mma_f16(cl[0][0], ah0, ah1, ah2, ah3, b00, b01);
        mma_f16(cl[0][1], al0, al1, al2, al3, b00, b01);
        mma_f16(cl[1][0], ah0, ah1, ah2, ah3, b10, b11);
        mma_f16(cl[1][1], al0, al1, al2, al3, b10, b11);
      }
#pragma unroll
      for (int ks = kF8L / 16; ks < kF8W / 16; ++ks) {
        uint32_t ah0, ah1, ah2, ah3, al0, al1, al2, al3, b00, b01, b10, b11;
        ldsm_x4(qhi_a + q_lane + 32 * ks, ah0, ah1, ah2, ah3);
        ldsm_x4(qlo_a + q_lane + 32 * ks, al0, al1, al2, al3);
        ldsm_x4(ks_lane + 32 * ks, b00, b01, b10, b11);
        mma_f16(cr[0][0], ah0, ah1, ah2, ah3, b00, b01);
        mma_f16(cr[0][1], al0, al1, al2, al3, b00, b01);
        mma_f16(cr[1][0], ah0, ah1, ah2, ah3, b10, b11);
        mma_f16(cr[1][1], al0, al1, al2, al3, b10, b11);
      }
      // C fragment of (f): rows (heads) g, g + 8; columns (tokens) 16 nq + 8 f + 2t, + 1
      float sc[2][4];
#pragma unroll
      for (int f = 0; f < 2; ++f) {
        const int kc = 16 * nq + 8 * f + 2 * t;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float l = cl[f][0][i] + cl[f][1][i], r = cr[f][0][i] + cr[f][1][i];
          float v = fmaf(ls[f][i & 1], l, rs[f][i & 1] * r);
          if (kc + (i & 1) >= nvalid) v = -INFINITY;
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
            pack_half2(p0 * ls[f][0], p1 * ls[f][1]);
        *reinterpret_cast<uint32_t*>(sm.p + (mb * 16 + g + 8) * kF8PStride + 2 * kc) =
            pack_half2(p2 * ls[f][0], p3 * ls[f][1]);
      }
      z_part[0] = fmaf(z_part[0], c0, zs0);
      z_part[1] = fmaf(z_part[1], c1, zs1);
      if (nq == 0 && t == 0) {
        sm.corr[mb * 16 + g] = c0;
        sm.corr[mb * 16 + g + 8] = c1;
      }
      consumers_sync();

      // ---------------- context: O[32 heads][dims 64 warp ..] += P' . latent
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
#pragma unroll
      for (int ks = 0; ks < kF8Keys / 16; ++ks) {
        uint32_t a0[4], a1[4];
        ldsm_x4(p_a + (0 * 16 + lrow) * kF8PStride + 16 * (2 * ks + lchunk), a0[0], a0[1], a0[2], a0[3]);
        ldsm_x4(p_a + (1 * 16 + lrow) * kF8PStride + 16 * (2 * ks + lchunk), a1[0], a1[1], a1[2], a1[3]);
#pragma unroll
        for (int nb = 0; nb < 8; nb += 2) {
          uint32_t b0, b1, b2, b3;  // (n-block nb: tokens 0-7, 8-15), (n-block nb + 1: tokens 0-7, 8-15)
          ldsm_x4_t(kv_lane + 16 * ks * kF8TStride + 16 * nb, b0, b1, b2, b3);
          mma_f16(acc[0][nb], a0[0], a0[1], a0[2], a0[3], b0, b1);
          mma_f16(acc[1][nb], a1[0], a1[1], a1[2], a1[3], b0, b1);
          mma_f16(acc[0][nb + 1], a0[0], a0[1], a0[2], a0[3], b2, b3);
          mma_f16(acc[1][nb + 1], a1[0], a1[1], a1[2], a1[3], b2, b3);
        }
      }
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
        float* dst = a.ws_acc + pi * kF8L + 64 * warp + 2 * t;
#pragma unroll
        for (int nb = 0; nb < 8; ++nb)
          *reinterpret_cast<float2*>(dst + 8 * nb) =
              bad ? make_float2(NAN, NAN) : make_float2(acc[x][nb][2 * hr], acc[x][nb][2 * hr + 1]);
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
    cudaError_t e = set_max_smem_once<decode_fp8_kernel<true>>((int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_fp8_kernel<true>, grid, dim3((kF8Warps + 1) * 32), smem, s, a);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = set_max_smem_once<decode_fp8_kernel<false>>((int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_fp8_kernel<false>, grid, dim3((kF8Warps + 1) * 32), smem, s, a);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace kvq
