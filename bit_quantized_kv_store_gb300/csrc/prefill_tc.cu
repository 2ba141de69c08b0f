// prefill_tc.cu -- causal prefill attention over decoded 4-bit slots on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Follows "qwen27 CUDA: an opt-in 4-bit attention cache (262K on a 24 GB card)",
// section "What it is": prompt chunks are packed into the cache, then attended
// with the prefill-attention kernel over decoded slots.  Query i of the chunk
// sits at absolute position q_start + i and attends keys 0 .. q_start + i, in the
// rotated space; the output is rotated back.
//
// One CTA per (block of 128/g query positions x the g query heads of a GQA group,
// KV head): M = 128 rows (row = iq * g + h), so every decoded key/value tile
// serves the whole group.  Keys are processed in tiles of 64.  Warp roles:
//  * warps 0, 2   producers of the raw 4-bit K pages (warp 0) and V pages (warp
//                 2), each into its own 2-stage ring so that neither side waits
//                 for the other -- codes by 2-D TMA boxes of 16 rows with the
//                 128-byte swizzle, scales by 1-D bulk copies;
//  * warp 1       MMA issuer (one thread) and tensor-memory owner;
//  * warps 4..7   softmax: one tensor-memory lane (= one row) per thread; they
//                 also rotate and split the queries at the start and normalise,
//                 rotate back and store the output at the end;
//  * warps 8, 9, 12, 13   decode K exactly as the sum of two f16 terms
//                 K_a = f16((c-8)s), K_b = (c-8)s - K_a (exact), written by
//                 stmatrix, in two halves of 128 dims so that the next tile's
//                 first half is decoded while the tensor cores still read the
//                 second half;
//  * warps 10, 11, 14, 15 decode V: f16((c-8)s), written transposed (keys
//                 contiguous per value dim) by stmatrix.trans.
// Warp w runs on SM sub-partition w % 4, so each sub-partition holds a softmax
// warp and decoders of one kind only; the decoders' and the softmax's loops are
// kept rolled (16-column / 8-key steps) so that the four roles' code sharing a
// sub-partition stays small -- with every loop unrolled, instruction fetch
// starved all roles.
// Each decoder lane reads one 16- or 8-byte chunk of a key row and produces the
// (row = key, two adjacent dims) fragment of 8x8 matrices; the stores fill whole
// 128-byte core matrices, so neither side has shared-memory bank conflicts.
// Scores S = q_hi.K_a + q_hi.K_b + q_lo.K_a (q split into f16 high and low
// parts, ~22 bits; q_hi is the A operand from tensor memory, q_lo from shared
// memory) accumulate in one of two tensor-memory S buffers, so the scores of
// tile j+1 are computed while the softmax works on tile j (the softmax reads S
// twice from tensor memory, for the maximum and for the exponentials, 16
// columns at a time).  P (f16) goes to
// shared memory and P.V accumulates into O (128 x 256 f32, tensor memory); the
// MMA issuer runs P.V of tile j after the scores of tile j+1.  The softmax
// rescales O lazily, only when the running maximum grows by more than 8 (base
// 2), so P stays <= 256.
#include "kernels.cuh"
#include "tc05.cuh"

namespace kvq {

constexpr int kPfKeys = 64;
constexpr int kPfStages = 2;
constexpr int kPfThreads = 512;
constexpr int kPfDim = 256;

// tensor-memory columns (512 allocated)
constexpr uint32_t kTmQhi = 0;  // 128 columns: q high part, f16 pairs (row = lane)
constexpr uint32_t kTmS = 128;  // 2 x 64 columns: scores of even / odd tiles, f32
constexpr uint32_t kTmO = 256;  // 256 columns: output accumulator, f32

struct __align__(1024) PfRaw {  // one 64-key tile of raw K or V cache rows (4 pages of 16 slots)
  uint8_t codes[64 * 128];       // 128-byte swizzled per 16-row page (chunk c of row r at c ^ (r & 7))
  uint16_t scales[64 * 8];
};
static_assert(sizeof(PfRaw) == 9216, "raw stage size");

struct PfSmem {
  PfRaw rawk[kPfStages];
  PfRaw rawv[kPfStages];
  // UMMA K-major layouts, 8-row x 16-byte core matrices:
  //   qlo, ka, kb: element (row, d) at (row/8)*4096 + (d/8)*128 + (row%8)*16 + (d%8)*2
  //   vt:          element (d, key) at (d/8)*1024 + (key/8)*128 + (d%8)*16 + (key%8)*2
  //   p:           element (row, key) at (row/8)*1024 + (key/8)*128 + (row%8)*16 + (key%8)*2
  uint8_t qlo[128 * kPfDim * 2];
  uint8_t ka[kPfKeys * kPfDim * 2];
  uint8_t kb[kPfKeys * kPfDim * 2];
  uint8_t vt[kPfDim * kPfKeys * 2];
  uint8_t p[128 * kPfKeys * 2];
  uint64_t rawk_full[kPfStages], rawk_empty[kPfStages];
  uint64_t rawv_full[kPfStages], rawv_empty[kPfStages];
  uint64_t k_ready[2], k_free[2];  // per half of the head dims
  uint64_t s_full[2], s_free[2];   // per S buffer
  uint64_t v_ready, p_full, pv_done, drained;
  uint32_t tmem_base;
  int abort;
  int poison;
};
static_assert(sizeof(PfSmem) + 1024 <= 232448, "prefill shared memory exceeds the 227 KB per-CTA limit");

// Bounded wait shared by the roles: gives up on the CTA-wide abort flag or after
// ~2 s (then raises the flag and KVQ_DEV_TIMEOUT) so that no role can hang.
__device__ __forceinline__ bool pf_wait(PfSmem& sm, uint64_t* bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 31u) {
      if (*reinterpret_cast<volatile int*>(&sm.abort)) return false;
      if (global_timer_ns() - t0 > 2000000000ull) {
        atomicExch(&sm.abort, 1);
        set_status(status, KVQ_DEV_TIMEOUT);
        return false;
      }
    }
  }
}

// One arrival per warp: every lane has ordered its own accesses (generic ->
// async-proxy fence, or tcgen05 fence) before calling; the warp converges and
// lane 0 arrives, so a barrier counts warps, not threads.
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Warp-uniform form of pf_wait for roles that issue warp-collective instructions.
__device__ __forceinline__ bool pf_wait_warp(PfSmem& sm, uint64_t* bar, uint32_t parity, int32_t* status) {
  return __all_sync(0xffffffffu, pf_wait(sm, bar, parity, status));
}

__device__ __forceinline__ void tma_rows_2d(void* dst, const CUtensorMap* map, int row, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(smem_u32(bar))
      : "memory");
}

// In-register 32-point Walsh-Hadamard butterfly (stages 1, 2, 4, 8, 16), no scaling.
__device__ __forceinline__ void fwht32_regs(float (&x)[32]) {
#pragma unroll
  for (int h = 1; h < 32; h <<= 1)
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if ((i & h) == 0) {
        const float u = x[i], v = x[i + h];
        x[i] = u + v;
        x[i + h] = u - v;
      }
}

// shared-memory loads at a 32-bit shared address
__device__ __forceinline__ uint4 pf_lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint2 pf_lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint32_t word_at(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// One stored code byte of w (element d in the low nibble, d+1 in the high
// nibble; `prmt_sel` picks the byte) -> the exact f16 pair (c_d - 8, c_{d+1} - 8).
// prmt copies the byte to bytes 0 and 2; the lop3 keeps the low nibble in the low
// half and the high nibble (times 16) in the high half under the f16 exponent of
// 1024; the hfma2 maps 1024 + c -> c - 8 and 1024 + 16c -> c - 8, exactly.
__device__ __forceinline__ __half2 code_pair(uint32_t w, uint32_t prmt_sel) {
  const uint32_t x = and_or(prmt(w, 0u, prmt_sel), 0x00F0000Fu, 0x64006400u);
  return __hfma2(u32_as_h2(x), u32_as_h2(0x2C003C00u) /* (1, 1/16) */, u32_as_h2(0xD480E408u) /* (-1032, -72) */);
}

// prmt selector copying byte `b` of the first operand to bytes 0 and 2 (zeros elsewhere).
__host__ __device__ constexpr uint32_t spread_sel(uint32_t b) { return 0x4040u | b | (b << 8); }

// (s, s) from the f16 scale in half `hi` of word w.
__device__ __forceinline__ __half2 scale_pair(uint32_t w, int hi) {
  return u32_as_h2(prmt(w, w, hi ? 0x3232u : 0x1010u));
}

__global__ void __launch_bounds__(kPfThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillArgs a) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  PfSmem& sm = *reinterpret_cast<PfSmem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = blockIdx.x, kvh = blockIdx.y;
  const kvq_cache& c = a.c;
  const int grp = a.group;
  const int qpb = 128 / grp;  // query positions per CTA
  const int q0 = qb * qpb;
  const int nq_blk = min(qpb, a.n_q - q0);
  const int kmax = a.q_start + q0 + nq_blk;  // keys [0, kmax)
  const int ntiles = (kmax + kPfKeys - 1) / kPfKeys;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPfStages; ++s) {
      mbar_init(&sm.rawk_full[s], 1);
      mbar_init(&sm.rawk_empty[s], 4);  // one arrival per K-decoder warp
      mbar_init(&sm.rawv_full[s], 1);
      mbar_init(&sm.rawv_empty[s], 4);  // one arrival per V-decoder warp
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sm.k_ready[h], 4);
      mbar_init(&sm.k_free[h], 1);
      mbar_init(&sm.s_full[h], 1);
      mbar_init(&sm.s_free[h], 4);
    }
    mbar_init(&sm.v_ready, 4);
    mbar_init(&sm.p_full, 4);
    mbar_init(&sm.pv_done, 1);
    mbar_init(&sm.drained, 1);
    sm.abort = 0;
    sm.poison = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&sm.tmem_base, 512);
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = sm.tmem_base;
  const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;

  if (warp >= 4 && warp < 8) {
    // ---------------- queries: rotate, scale, split; q_hi -> TMEM, q_lo -> smem
    const int r = 32 * (warp - 4) + lane;
    const int iq = r / grp, h = r % grp;
    const bool valid = (r < qpb * grp) && (iq < nq_blk);
    const int64_t qrow = ((int64_t)(q0 + iq) * a.Hq + kvh * grp + h) * kPfDim;
    for (int G = 0; G < 8; ++G) {
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float v = 0.f;
        if (valid)
          v = a.dtype == KVQ_DT_F32 ? static_cast<const float*>(a.q)[qrow + 32 * G + i]
                                    : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[qrow + 32 * G + i]);
        x[i] = v;
      }
      const bool rot = a.rotate != 0;  // Q4_0: the query as given
      if (rot) fwht32_regs(x);
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float x0 = (rot ? __fmul_rn(x[2 * i], kHadamardScale) : x[2 * i]) * a.qscale;
        const float x1 = (rot ? __fmul_rn(x[2 * i + 1], kHadamardScale) : x[2 * i + 1]) * a.qscale;
        split_f16(x0, x1, hi[i], lo[i]);
      }
      __syncwarp();  // the tensor-memory store is warp-collective
      tmem_st16(tbase + lane_off + kTmQhi + 16 * G, hi);
      uint8_t* dst = sm.qlo + (r / 8) * 4096 + (r % 8) * 16;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
        *reinterpret_cast<uint4*>(dst + (4 * G + cc) * 128) =
            make_uint4(lo[4 * cc], lo[4 * cc + 1], lo[4 * cc + 2], lo[4 * cc + 3]);
    }
    tmem_wait_st();
    fence_proxy_async();
    tc_fence_before();
  }
  __syncthreads();  // queries ready (TMEM and shared memory)
  tc_fence_after();

  if (warp == 0 || warp == 2) {
    // ---------------- producers: K pages (warp 0), V pages (warp 2)
    if (lane == 0) {
      const bool is_k = warp == 0;
      const CUtensorMap* map = is_k ? &a.tm_k : &a.tm_v;
      const uint16_t* scales = static_cast<const uint16_t*>(is_k ? c.k_scale : c.v_scale);
      PfRaw* ring = is_k ? sm.rawk : sm.rawv;
      uint64_t* full = is_k ? sm.rawk_full : sm.rawv_full;
      uint64_t* empty = is_k ? sm.rawk_empty : sm.rawv_empty;
      const int32_t* bt = a.block_table;
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % kPfStages;
        if (!pf_wait(sm, &empty[s], ((j / kPfStages) & 1) ^ 1, a.status)) break;
        PfRaw& st = ring[s];
        int64_t rows[4];
        uint32_t bytes = 0;
        for (int pg = 0; pg < 4; ++pg) {
          rows[pg] = -1;
          const int key0 = j * kPfKeys + 16 * pg;
          if (key0 >= kmax) continue;
          const int32_t page = bt[key0 / c.page_size];
          if (page < 0 || page >= c.num_pages) {
            set_status(a.status, KVQ_DEV_BAD_PAGE);
            sm.poison = 1;
            continue;
          }
          rows[pg] = ((int64_t)page * c.num_kv_heads + kvh) * c.page_size + key0 % c.page_size;
          bytes += 16 * 128 + 16 * 16;
        }
        if (bytes == 0) {
          mbar_arrive(&full[s]);
          continue;
        }
        mbar_arrive_expect_tx(&full[s], bytes);
        for (int pg = 0; pg < 4; ++pg) {
          if (rows[pg] < 0) continue;
          tma_rows_2d(st.codes + pg * 2048, map, static_cast<int>(rows[pg]), &full[s]);
          bulk_g2s(st.scales + pg * 128, scales + rows[pg] * 8, 256, &full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer: QK(j) into S[j % 2], then PV(j - 1)
    // Descriptors are built once; a k-step of 16 advances every operand by 256
    // bytes (16 in descriptor units) and the q_hi columns by 8, so the unrolled
    // runs below issue one instruction per MMA.
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_f16_f32(128, kPfKeys);
      constexpr uint32_t id_pv = idesc_f16_f32(128, kPfDim);
      const uint64_t dka = umma_desc(smem_u32(sm.ka), 128, 4096), dkb = umma_desc(smem_u32(sm.kb), 128, 4096);
      const uint64_t dql = umma_desc(smem_u32(sm.qlo), 128, 4096);
      const uint64_t dp = umma_desc(smem_u32(sm.p), 128, 1024), dvt = umma_desc(smem_u32(sm.vt), 128, 1024);
      const uint32_t tq = tbase + kTmQhi;
      bool ok = true;
      for (int j = 0; j <= ntiles && ok; ++j) {
        if (j < ntiles) {
          const int b = j & 1;
          const uint32_t sacc = tbase + kTmS + 64 * b;
          // softmax(j - 2) has read S[b]
          if (j >= 2 && !pf_wait(sm, &sm.s_free[b], ((j >> 1) - 1) & 1, a.status)) break;
          // first half of the head dims: k-steps 0..7
          if (!pf_wait(sm, &sm.k_ready[0], j & 1, a.status)) break;
          tc_fence_after();
          umma_ts(sacc, tq, dka, id_qk, 0u);
          umma_ts_acc(sacc, tq, dkb, id_qk);
          umma_ss_acc(sacc, dql, dka, id_qk);
#pragma unroll
          for (int s = 1; s < 8; ++s) {
            umma_ts_acc(sacc, tq + 8 * s, dka + 16 * s, id_qk);
            umma_ts_acc(sacc, tq + 8 * s, dkb + 16 * s, id_qk);
            umma_ss_acc(sacc, dql + 16 * s, dka + 16 * s, id_qk);
          }
          umma_commit(&sm.k_free[0]);
          // second half: k-steps 8..15
          if (!pf_wait(sm, &sm.k_ready[1], j & 1, a.status)) break;
          tc_fence_after();
#pragma unroll
          for (int s = 8; s < 16; ++s) {
            umma_ts_acc(sacc, tq + 8 * s, dka + 16 * s, id_qk);
            umma_ts_acc(sacc, tq + 8 * s, dkb + 16 * s, id_qk);
            umma_ss_acc(sacc, dql + 16 * s, dka + 16 * s, id_qk);
          }
          umma_commit(&sm.k_free[1]);
          umma_commit(&sm.s_full[b]);
        }
        if (j >= 1) {  // P.V of tile j - 1
          const int jp = j - 1;
          if (!pf_wait(sm, &sm.p_full, jp & 1, a.status)) break;
          if (!pf_wait(sm, &sm.v_ready, jp & 1, a.status)) break;
          tc_fence_after();
          umma_ss(tbase + kTmO, dp, dvt, id_pv, jp > 0 ? 1u : 0u);
#pragma unroll
          for (int s = 1; s < kPfKeys / 16; ++s) umma_ss_acc(tbase + kTmO, dp + 16 * s, dvt + 16 * s, id_pv);
          umma_commit(&sm.pv_done);
        }
      }
      // every MMA issued so far has finished before tensor memory is released
      // (bounded, and independent of the abort flag)
      umma_commit(&sm.drained);
      mbar_wait_bounded(&sm.drained, 0);
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- softmax, one row per thread
    const int r = 32 * (warp - 4) + lane;
    const int iq = r / grp, h = r % grp;
    const bool valid = (r < qpb * grp) && (iq < nq_blk);
    const int qpos = a.q_start + q0 + iq;  // keys 0 .. qpos
    uint8_t* prow = sm.p + (r >> 3) * 1024 + (r & 7) * 16;
    // tcgen05.ld/st are warp-collective (.sync.aligned): every branch around
    // them is made warp-uniform, including the failure paths.
    float m_run = -INFINITY, z = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      const int b = j & 1;
      ok = pf_wait_warp(sm, &sm.s_full[b], (j >> 1) & 1, a.status);
      if (!ok) break;
      tc_fence_after();
      const uint32_t sadr = tbase + lane_off + kTmS + 64 * b;
      const int lim = valid ? qpos - j * kPfKeys : -1;  // keys i <= lim of this tile are visible
      // pass 1: the row maximum over the visible keys, 16 columns at a time
      float tmax = -INFINITY;
#pragma unroll 1
      for (int cc = 0; cc < kPfKeys / 16; ++cc) {
        uint32_t v[16];
        tmem_ld16(sadr + 16 * cc, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) tmax = fmaxf(tmax, (16 * cc + i > lim) ? -INFINITY : __uint_as_float(v[i]));
      }
      // Raise a row's reference maximum only when its scores grew by more than 8
      // (base 2); rows that rescale multiply their accumulated O and z by corr.
      const bool raise = tmax > m_run + 8.f;
      float corr = 1.f;
      if (raise) {
        corr = (m_run == -INFINITY) ? 1.f : fast_exp2(m_run - tmax);  // O and z are still zero at -inf
        z *= corr;
        m_run = tmax;
      }
      const float mu = (m_run == -INFINITY) ? 0.f : m_run;
      if (j > 0) {  // PV(j-1) must be done: it reads P and accumulates into O
        ok = pf_wait_warp(sm, &sm.pv_done, (j - 1) & 1, a.status);
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, raise && corr != 1.f)) {  // warp-uniform O rescale
#pragma unroll 1
          for (int cc = 0; cc < kPfDim / 16; ++cc) {
            uint32_t o[16];
            tmem_ld16(tbase + lane_off + kTmO + 16 * cc, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
            tmem_st16(tbase + lane_off + kTmO + 16 * cc, o);
          }
          tmem_wait_st();
        }
      }
      // pass 2: p = 2^(s - mu) (0 for masked keys), f16 pairs into P, 16 keys at a time
      float zs = 0.f;
#pragma unroll 1
      for (int cc = 0; cc < kPfKeys / 16; ++cc) {
        uint32_t v[16], pk[8];
        tmem_ld16(sadr + 16 * cc, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float p0 = (16 * cc + 2 * i > lim) ? 0.f : fast_exp2(__uint_as_float(v[2 * i]) - mu);
          const float p1 = (16 * cc + 2 * i + 1 > lim) ? 0.f : fast_exp2(__uint_as_float(v[2 * i + 1]) - mu);
          zs += p0 + p1;
          pk[i] = pack_half2(p0, p1);
        }
        *reinterpret_cast<uint4*>(prow + (2 * cc) * 128) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(prow + (2 * cc + 1) * 128) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      }
      z += zs;
      tc_fence_before();
      warp_arrive(&sm.s_free[b], lane);  // S[b] read
      fence_proxy_async();
      warp_arrive(&sm.p_full, lane);
    }
    // ---------------- epilogue: O / z, rotate back, store
    if (ok) ok = pf_wait_warp(sm, &sm.pv_done, (ntiles - 1) & 1, a.status);
    if (ok) {
      tc_fence_after();
      const bool bad = sm.poison != 0 || sm.abort != 0;
      const float inv = (z > 0.f) ? 1.f / z : 0.f;
      for (int G = 0; G < 8; ++G) {
        uint32_t o[32];
        __syncwarp();  // reconverge after the previous iteration's per-row store
        tmem_ld32(tbase + lane_off + kTmO + 32 * G, o);
        tmem_wait_ld();
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(o[i]) * inv;
        const bool rot = a.rotate != 0;  // Q4_0: nothing to rotate back
        if (rot) {
          fwht32_regs(x);
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __fmul_rn(x[i], kHadamardScale);
        }
        if (valid) {
          float* dst = a.out + ((int64_t)(q0 + iq) * a.Hq + kvh * grp + h) * kPfDim + 32 * G;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) =
                bad ? make_float4(NAN, NAN, NAN, NAN) : make_float4(x[i], x[i + 1], x[i + 2], x[i + 3]);
        }
      }
    }
  } else if (warp >= 8 && (warp & 2) == 0) {
    // ---------------- K decoder (warps 8, 9, 12, 13): key blocks 2kw, 2kw+1 of every tile, by halves
    const int kw = (warp & 1) + 2 * ((warp - 8) >> 2);
    const int krow = lane >> 2;  // key within the 8-key block
    // byte lane & 3 of word m of a group's 16 bytes: elements 8m + 2 (lane & 3), + 1
    const uint32_t sel_b = spread_sel(lane & 3);
    const uint32_t ka = smem_u32(sm.ka), kbuf = smem_u32(sm.kb);
    // stmatrix row address: matrix lane / 8 of the four (group 4 half + lane / 8), its row lane % 8
    const uint32_t st_off = (uint32_t)(lane >> 3) * 4 * 128 + (uint32_t)(lane & 7) * 16;
    bool ok = true;
    for (int j = 0; j < ntiles && ok; ++j) {
      const int s = j % kPfStages;
      if (!pf_wait_warp(sm, &sm.rawk_full[s], (j / kPfStages) & 1, a.status)) break;
      const uint32_t st_codes = smem_u32(sm.rawk[s].codes), st_scales = smem_u32(sm.rawk[s].scales);
      const int jk0 = j * kPfKeys;
      for (int half = 0; half < 2; ++half) {
        // QK(j-1) has read this half of K_a, K_b
        if (j > 0 && !pf_wait_warp(sm, &sm.k_free[half], (j - 1) & 1, a.status)) {
          ok = false;
          break;
        }
#pragma unroll 1
        for (int kbl = 0; kbl < 2; ++kbl) {
          const int kbk = 2 * kw + kbl;
          const int key = 8 * kbk + krow;
          // scales of groups 4 half .. 4 half + 3 (zero past kmax: stale codes give zero)
          uint2 sc = pf_lds64(st_scales + key * 16 + 8 * half);
          if (jk0 + key >= kmax) sc = make_uint2(0, 0);
          const __half2 s2[4] = {scale_pair(sc.x, 0), scale_pair(sc.x, 1), scale_pair(sc.y, 0), scale_pair(sc.y, 1)};
          // the key's code blocks of groups 4 half .. 4 half + 3 (16-byte chunk G of the row)
          uint4 wg[4];
#pragma unroll
          for (int gl = 0; gl < 4; ++gl) wg[gl] = pf_lds128(st_codes + key * 128 + (((4 * half + gl) ^ (key & 7)) << 4));
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            uint32_t va[4], vb[4];
#pragma unroll
            for (int gl = 0; gl < 4; ++gl) {
              const __half2 cv = code_pair(word_at(wg[gl], m), sel_b);
              const __half2 xa = __hmul2(cv, s2[gl]);
              va[gl] = h2_as_u32(xa);
              vb[gl] = h2_as_u32(__hfma2(cv, s2[gl], __hneg2(xa)));  // exact remainder
            }
            // matrix (G = 4 half + gl, m): key block kbk, d-block 4G + m
            const uint32_t off = (uint32_t)kbk * 4096 + (uint32_t)(16 * half + m) * 128 + st_off;
            stmatrix_x4(ka + off, va[0], va[1], va[2], va[3]);
            stmatrix_x4(kbuf + off, vb[0], vb[1], vb[2], vb[3]);
          }
        }
        fence_proxy_async();
        warp_arrive(&sm.k_ready[half], lane);
      }
      if (ok) warp_arrive(&sm.rawk_empty[s], lane);
    }
  } else if (warp >= 8) {
    // ---------------- V decoder (warps 10, 11, 14, 15): key blocks 2vw, 2vw+1 of every tile
    const int vw = (warp & 1) + 2 * ((warp - 10) >> 2);
    const int krow = lane >> 2;
    const uint32_t sel_b = spread_sel(lane & 3);  // as in the K decoder
    const uint32_t vt = smem_u32(sm.vt);
    // stmatrix row address: matrix lane / 8 of the four (group G), its row lane % 8
    const uint32_t st_off = (uint32_t)(lane >> 3) * 4 * 1024 + (uint32_t)(lane & 7) * 16;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kPfStages;
      if (!pf_wait_warp(sm, &sm.rawv_full[s], (j / kPfStages) & 1, a.status)) break;
      if (j > 0 && !pf_wait_warp(sm, &sm.pv_done, (j - 1) & 1, a.status)) break;  // PV(j-1) is done with vt
      const uint32_t st_codes = smem_u32(sm.rawv[s].codes), st_scales = smem_u32(sm.rawv[s].scales);
      const int jk0 = j * kPfKeys;
#pragma unroll 1
      for (int kbl = 0; kbl < 2; ++kbl) {
        const int kbk = 2 * vw + kbl;
        const int key = 8 * kbk + krow;
        uint4 sc = pf_lds128(st_scales + key * 16);
        if (jk0 + key >= kmax) sc = make_uint4(0, 0, 0, 0);  // zero scale past kmax: stale codes give zero
        __half2 s2[8];
#pragma unroll
        for (int G = 0; G < 8; ++G) s2[G] = scale_pair(word_at(sc, G >> 1), G & 1);
        uint4 wg[8];  // the key's 8 code blocks (16-byte chunk G of the row)
#pragma unroll
        for (int G = 0; G < 8; ++G) wg[G] = pf_lds128(st_codes + key * 128 + ((G ^ (key & 7)) << 4));
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint32_t v[8];
#pragma unroll
          for (int G = 0; G < 8; ++G) v[G] = h2_as_u32(__hmul2(code_pair(word_at(wg[G], m), sel_b), s2[G]));
          // matrix (G, m): d-block 4G + m, key block kbk -> vt + (4G + m) * 1024 + kbk * 128
          const uint32_t base = vt + (uint32_t)m * 1024 + (uint32_t)kbk * 128 + st_off;
          stmatrix_x4_trans(base, v[0], v[1], v[2], v[3]);
          stmatrix_x4_trans(base + 16 * 1024, v[4], v[5], v[6], v[7]);
        }
      }
      fence_proxy_async();
      warp_arrive(&sm.v_ready, lane);
      warp_arrive(&sm.rawv_empty[s], lane);
    }
  }

  pdl_trigger();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
  if (a.n_q == 0) return cudaSuccess;
  const size_t smem = sizeof(PfSmem) + 1024;
  cudaError_t e = set_max_smem_once<prefill_tc_kernel>(static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int qpb = 128 / a.group;
  dim3 grid((a.n_q + qpb - 1) / qpb, a.c.num_kv_heads);
  e = launch_pdl(prefill_tc_kernel, grid, dim3(kPfThreads), smem, s, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvq
