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
//  * warp 0       producer: the raw 4-bit pages into a 2-stage ring -- codes by
//                 2-D TMA boxes of 16 rows with the 128-byte swizzle (so the
//                 decoders' shared-memory reads spread over the banks), scales
//                 by 1-D bulk copies;
//  * warp 1       MMA issuer (one thread) and tensor-memory owner;
//  * warps 4..7   softmax: one tensor-memory lane (= one row) per thread; they
//                 also rotate and split the queries at the start and normalise,
//                 rotate back and store the output at the end;
//  * warps 8..11  decode the tile: K exactly as the sum of two f16 terms
//                 K_a = f16((c-8)s), K_b = (c-8)s - K_a (exact), V as
//                 f16((c-8)s) stored transposed (keys contiguous per value dim).
// Scores S = q_hi.K_a + q_hi.K_b + q_lo.K_a (q split into f16 high and low
// parts, ~22 bits; q_hi is the A operand from tensor memory, q_lo from shared
// memory) accumulate in tensor memory; P (f16) is written back to tensor memory
// and P.V accumulates into O (128 x 256 f32, tensor memory).  The softmax
// rescales O lazily, only when the running maximum grows by more than 8 (base 2),
// so P stays <= 256.
#include "kernels.cuh"
#include "tc05.cuh"

namespace kvq {

constexpr int kPfKeys = 64;
constexpr int kPfStages = 2;
constexpr int kPfThreads = 384;
constexpr int kPfDim = 256;

// tensor-memory columns (512 allocated)
constexpr uint32_t kTmQhi = 0;    // 128 columns: q high part, f16 pairs (row = lane)
constexpr uint32_t kTmS = 128;    // 64 columns: scores, f32
constexpr uint32_t kTmP = 192;    // 32 columns: probabilities, f16 pairs
constexpr uint32_t kTmO = 256;    // 256 columns: output accumulator, f32

struct __align__(1024) PfRaw {  // one 64-key tile of raw cache rows (4 pages of 16 slots)
  uint8_t kc[64 * 128];          // K codes, 128-byte swizzled per 16-row page (chunk c of row r at c ^ (r & 7))
  uint8_t vc[64 * 128];          // V codes, same
  uint16_t ks[64 * 8];
  uint16_t vs[64 * 8];
};
static_assert(sizeof(PfRaw) == 18432, "raw stage size");

struct PfSmem {
  PfRaw raw[kPfStages];
  // UMMA K-major layouts, 8-row x 16-byte core matrices:
  //   qlo, ka, kb: element (row, d) at (row/8)*4096 + (d/8)*128 + (row%8)*16 + (d%8)*2
  //   vt:          element (d, key) at (d/8)*1024 + (key/8)*128 + (d%8)*16 + (key%8)*2
  uint8_t qlo[128 * kPfDim * 2];
  uint8_t ka[kPfKeys * kPfDim * 2];
  uint8_t kb[kPfKeys * kPfDim * 2];
  uint8_t vt[kPfDim * kPfKeys * 2];
  uint64_t raw_full[kPfStages];
  uint64_t raw_empty[kPfStages];
  uint64_t k_ready, v_ready, s_full, p_full, pv_done;
  uint32_t tmem_base;
  int abort;
  int poison;
};

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

__device__ __forceinline__ void tma_rows_2d(void* dst, const CUtensorMap* map, int row, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint32_t bias_pair(uint32_t x) {  // (1024 + c) pair -> (c - 8) pair, exact
  return h2_as_u32(__hsub2(u32_as_h2(x), u32_as_h2(0x64086408u)));
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

__global__ void __launch_bounds__(kPfThreads, 1) prefill_tc_kernel(const __grid_constant__ PrefillArgs a) {
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
      mbar_init(&sm.raw_full[s], 1);
      mbar_init(&sm.raw_empty[s], 128);
    }
    mbar_init(&sm.k_ready, 128);
    mbar_init(&sm.v_ready, 128);
    mbar_init(&sm.s_full, 1);
    mbar_init(&sm.p_full, 128);
    mbar_init(&sm.pv_done, 1);
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
      fwht32_regs(x);
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float x0 = __fmul_rn(x[2 * i], kHadamardScale) * a.qscale;
        const float x1 = __fmul_rn(x[2 * i + 1], kHadamardScale) * a.qscale;
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

  if (warp == 0) {
    // ---------------- producer
    if (lane == 0) {
      const int32_t* bt = a.block_table;
      for (int j = 0; j < ntiles; ++j) {
        const int s = j % kPfStages;
        if (!pf_wait(sm, &sm.raw_empty[s], ((j / kPfStages) & 1) ^ 1, a.status)) break;
        PfRaw& st = sm.raw[s];
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
          bytes += 2 * 16 * 128 + 2 * 16 * 16;
        }
        if (bytes == 0) {
          mbar_arrive(&sm.raw_full[s]);
          continue;
        }
        mbar_arrive_expect_tx(&sm.raw_full[s], bytes);
        for (int pg = 0; pg < 4; ++pg) {
          if (rows[pg] < 0) continue;
          tma_rows_2d(st.kc + pg * 2048, &a.tm_k, static_cast<int>(rows[pg]), &sm.raw_full[s]);
          tma_rows_2d(st.vc + pg * 2048, &a.tm_v, static_cast<int>(rows[pg]), &sm.raw_full[s]);
          bulk_g2s(st.ks + pg * 128, static_cast<const uint16_t*>(c.k_scale) + rows[pg] * 8, 256, &sm.raw_full[s]);
          bulk_g2s(st.vs + pg * 128, static_cast<const uint16_t*>(c.v_scale) + rows[pg] * 8, 256, &sm.raw_full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_f16_f32(128, kPfKeys);
      constexpr uint32_t id_pv = idesc_f16_f32(128, kPfDim);
      const uint32_t qlo = smem_u32(sm.qlo), ka = smem_u32(sm.ka), kb = smem_u32(sm.kb), vt = smem_u32(sm.vt);
      for (int j = 0; j < ntiles; ++j) {
        if (!pf_wait(sm, &sm.k_ready, j & 1, a.status)) break;
        tc_fence_after();
        for (int s = 0; s < kPfDim / 16; ++s) {
          const uint64_t da = umma_desc(ka + s * 256, 128, 4096);
          const uint64_t db = umma_desc(kb + s * 256, 128, 4096);
          umma_ts(tbase + kTmS, tbase + kTmQhi + 8 * s, da, id_qk, s > 0 ? 1u : 0u);
          umma_ts(tbase + kTmS, tbase + kTmQhi + 8 * s, db, id_qk, 1u);
          umma_ss(tbase + kTmS, umma_desc(qlo + s * 256, 128, 4096), da, id_qk, 1u);
        }
        umma_commit(&sm.s_full);
        if (!pf_wait(sm, &sm.p_full, j & 1, a.status)) break;
        if (!pf_wait(sm, &sm.v_ready, j & 1, a.status)) break;
        tc_fence_after();
        for (int s = 0; s < kPfKeys / 16; ++s)
          umma_ts(tbase + kTmO, tbase + kTmP + 8 * s, umma_desc(vt + s * 256, 128, 1024), id_pv,
                  (j > 0 || s > 0) ? 1u : 0u);
        umma_commit(&sm.pv_done);
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- softmax, one row per thread
    const int r = 32 * (warp - 4) + lane;
    const int iq = r / grp, h = r % grp;
    const bool valid = (r < qpb * grp) && (iq < nq_blk);
    const int qpos = a.q_start + q0 + iq;  // keys 0 .. qpos
    // tcgen05.ld/st are warp-collective (.sync.aligned): every branch around
    // them is made warp-uniform, including the failure paths.
    float m_run = -INFINITY, z = 0.f;
    bool ok = true;
    for (int j = 0; j < ntiles; ++j) {
      ok = __all_sync(0xffffffffu, pf_wait(sm, &sm.s_full, j & 1, a.status));
      if (!ok) break;
      tc_fence_after();
      uint32_t s0[32], s1[32];
      tmem_ld32(tbase + lane_off + kTmS, s0);
      tmem_ld32(tbase + lane_off + kTmS + 32, s1);
      tmem_wait_ld();
      float sv[64];
      const int key0 = j * kPfKeys;
      float tmax = -INFINITY;
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        float v = __uint_as_float(i < 32 ? s0[i] : s1[i - 32]);
        if (!valid || key0 + i > qpos) v = -INFINITY;
        sv[i] = v;
        tmax = fmaxf(tmax, v);
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
      if (j > 0 && __any_sync(0xffffffffu, raise && corr != 1.f)) {  // warp-uniform O rescale
        ok = __all_sync(0xffffffffu, pf_wait(sm, &sm.pv_done, (j - 1) & 1, a.status));
        if (!ok) break;
        tc_fence_after();
        for (int cc = 0; cc < kPfDim / 32; ++cc) {
          uint32_t o[32];
          tmem_ld32(tbase + lane_off + kTmO + 32 * cc, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
          tmem_st32(tbase + lane_off + kTmO + 32 * cc, o);
        }
      }
      uint32_t pk[32];
      float zs = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p0 = (sv[2 * i] == -INFINITY) ? 0.f : fast_exp2(sv[2 * i] - m_run);
        const float p1 = (sv[2 * i + 1] == -INFINITY) ? 0.f : fast_exp2(sv[2 * i + 1] - m_run);
        zs += p0 + p1;
        pk[i] = pack_half2(p0, p1);
      }
      z += zs;
      tmem_st32(tbase + lane_off + kTmP, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&sm.p_full);
    }
    // ---------------- epilogue: O / z, rotate back, store
    if (ok) ok = __all_sync(0xffffffffu, pf_wait(sm, &sm.pv_done, (ntiles - 1) & 1, a.status));
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
        fwht32_regs(x);
        if (valid) {
          float* dst = a.out + ((int64_t)(q0 + iq) * a.Hq + kvh * grp + h) * kPfDim + 32 * G;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) =
                bad ? make_float4(NAN, NAN, NAN, NAN)
                    : make_float4(__fmul_rn(x[i], kHadamardScale), __fmul_rn(x[i + 1], kHadamardScale),
                                  __fmul_rn(x[i + 2], kHadamardScale), __fmul_rn(x[i + 3], kHadamardScale));
        }
      }
    }
  } else if (warp >= 8) {
    // ---------------- decode K and V tiles
    const int t = threadIdx.x - 256;
    for (int j = 0; j < ntiles; ++j) {
      const int s = j % kPfStages;
      if (!pf_wait(sm, &sm.raw_full[s], (j / kPfStages) & 1, a.status)) break;
      const PfRaw& st = sm.raw[s];
      // K: thread -> key kk = t/2, groups 4*(t%2) .. +3; K_a, K_b rows
      if (j > 0 && !pf_wait(sm, &sm.s_full, (j - 1) & 1, a.status)) break;  // QK(j-1) done with ka/kb
      {
        const int kk = t >> 1, gh = t & 1;
        const bool kv = j * kPfKeys + kk < kmax;
        // chunk h of the row holds half-words (h, G = 0..7); this thread needs G = 4gh .. 4gh+3
        uint2 w[8];
#pragma unroll
        for (int h = 0; h < 8; ++h)
          w[h] = *reinterpret_cast<const uint2*>(st.kc + kk * 128 + ((h ^ (kk & 7)) << 4) + 8 * gh);
        const uint2 sc = *reinterpret_cast<const uint2*>(st.ks + kk * 8 + 4 * gh);
        uint8_t* arow = sm.ka + (kk >> 3) * 4096 + (kk & 7) * 16;
        uint8_t* brow = sm.kb + (kk >> 3) * 4096 + (kk & 7) * 16;
#pragma unroll
        for (int gl = 0; gl < 4; ++gl) {
          const int G = 4 * gh + gl;
          const uint32_t sw = (gl >> 1) ? sc.y : sc.x;
          const uint32_t s16 = (gl & 1) ? (sw >> 16) : (sw & 0xFFFFu);
          const __half2 s2 = u32_as_h2(s16 | (s16 << 16));
#pragma unroll
          for (int hp = 0; hp < 4; ++hp) {  // half-words h = 2hp, 2hp+1 fill one 16-byte chunk
            uint32_t av[4], bv[4];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int h = 2 * hp + e;
              const uint32_t wd = (gl >> 1) ? w[h].y : w[h].x;  // half-words (h, G & ~1), (h, G | 1)
              const uint32_t hw = (wd >> (16 * (gl & 1))) & 0xFFFFu;
              const uint32_t x = hw | (hw << 12);
              const __half2 c01 = u32_as_h2(bias_pair(and_or(x, 0x000F000Fu, 0x64006400u)));
              const __half2 c23 = u32_as_h2(bias_pair(and_or(x >> 8, 0x000F000Fu, 0x64006400u)));
              const __half2 a01 = __hmul2(c01, s2), a23 = __hmul2(c23, s2);
              const __half2 b01 = __hfma2(c01, s2, __hneg2(a01)), b23 = __hfma2(c23, s2, __hneg2(a23));
              av[2 * e] = h2_as_u32(a01);
              av[2 * e + 1] = h2_as_u32(a23);
              bv[2 * e] = h2_as_u32(b01);
              bv[2 * e + 1] = h2_as_u32(b23);
            }
            const int chunk = 4 * G + hp;  // d = 32G + 8hp .. +8
            const uint4 A = kv ? make_uint4(av[0], av[1], av[2], av[3]) : make_uint4(0, 0, 0, 0);
            const uint4 B = kv ? make_uint4(bv[0], bv[1], bv[2], bv[3]) : make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(arow + chunk * 128) = A;
            *reinterpret_cast<uint4*>(brow + chunk * 128) = B;
          }
        }
      }
      fence_proxy_async();
      mbar_arrive(&sm.k_ready);
      // V: thread -> keys 8*kb8 .. +7, stored words wi and wi+16; writes V^T chunks
      if (j > 0 && !pf_wait(sm, &sm.pv_done, (j - 1) & 1, a.status)) break;  // PV(j-1) done with vt
      {
        const int kb8 = t >> 4, wi = t & 15;
        uint32_t vsw[8];  // V scale word (groups G, G+1) of each of the 8 keys, per stored word
#pragma unroll
        for (int ww = 0; ww < 2; ++ww) {
          const int wd = wi + 16 * ww;     // stored word: half-words 2wd, 2wd+1
          const int h = (2 * wd) >> 3, G = (2 * wd) & 7;  // G even
          uint32_t vw[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int key = 8 * kb8 + k;
            const bool kv = j * kPfKeys + key < kmax;
            vw[k] = *reinterpret_cast<const uint32_t*>(st.vc + key * 128 + (((wd >> 2) ^ (key & 7)) << 4) +
                                                        4 * (wd & 3));
            vsw[k] = kv ? *reinterpret_cast<const uint32_t*>(st.vs + key * 8 + G) : 0u;  // zero scale past kmax
          }
          // word bytes: [hw(G).b0, hw(G).b1, hw(G+1).b0, hw(G+1).b1]; byte X holds elements (lo, hi)
#pragma unroll
          for (int X = 0; X < 4; ++X) {
            const int Gx = G + (X >> 1);
            const int d_lo = 32 * Gx + 4 * h + 2 * (X & 1);  // element of the low nibble; d_lo+1 the high
            uint32_t lo4[4], hi4[4];
#pragma unroll
            for (int kp = 0; kp < 4; ++kp) {  // key pair (2kp, 2kp+1)
              const uint32_t x = prmt(vw[2 * kp], vw[2 * kp + 1], (X | (X << 4) | ((X + 4) << 8) | ((X + 4) << 12)));
              const uint32_t ssel = (X >> 1) ? 0x7632u : 0x5410u;
              const __half2 s2 = u32_as_h2(prmt(vsw[2 * kp], vsw[2 * kp + 1], ssel));
              lo4[kp] = h2_as_u32(__hmul2(u32_as_h2(nib_lo_pair(x)), s2));
              hi4[kp] = h2_as_u32(__hmul2(u32_as_h2(nib_hi_pair(x)), s2));
            }
            uint8_t* base = sm.vt + kb8 * 128;
            *reinterpret_cast<uint4*>(base + (d_lo >> 3) * 1024 + (d_lo & 7) * 16) =
                make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
            *reinterpret_cast<uint4*>(base + ((d_lo + 1) >> 3) * 1024 + ((d_lo + 1) & 7) * 16) =
                make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]);
          }
        }
      }
      fence_proxy_async();
      mbar_arrive(&sm.v_ready);
      mbar_arrive(&sm.raw_empty[s]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tbase, 512);
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, cudaStream_t s) {
  if (a.n_q == 0) return cudaSuccess;
  const size_t smem = sizeof(PfSmem) + 1024;
  cudaError_t e =
      cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int qpb = 128 / a.group;
  dim3 grid((a.n_q + qpb - 1) / qpb, a.c.num_kv_heads);
  prefill_tc_kernel<<<grid, kPfThreads, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
