// decode_bf16.cu -- split-T decode attention over the unrotated bf16 cache (the
// bytes-read comparison run), on the tensor cores.
//
// Follows "qwen27 CUDA: an opt-in 4-bit attention cache (262K on a 24 GB card)",
// section "What it is": the 4-bit cache is opt-in and the bf16 cache is the
// default it is compared against; same split-T structure (512-key partitions
// plus the tail, per-partition (m, z, acc) partials merged by log-sum-exp), no
// rotation.
//
// GB300 design: the structure of the 4-bit kernel with bf16 operands fed to
// mma.m16n8k16 directly.  One CTA (2 warps, 2 resident per SM) per (partition,
// KV head, sequence); warp w owns keys [256w, 256w + 256) in tiles of 16,
// streamed through a private 2-stage shared-memory ring: K and V rows (512 B)
// arrive as four 128-byte column boxes of 16 rows each by 2-D TMA with the
// 128-byte swizzle (dense), or row by row into 528-byte padded rows (gather).
//  * Scores: keys on M (A = K rows by ldmatrix), the <= 8 heads of the GQA group
//    on N (B = query fragments in shared memory, split into bf16 high and low
//    parts, ~16 bits); keys enter exactly.
//  * Context: value dims on M (A = V^T by ldmatrix.trans), heads on N (B = P^T,
//    transposed in registers by movmatrix, split into bf16 high and low parts).
//  * Base-2 online softmax per head; the 2 warps' partials are combined in
//    shared memory.
#include "kernels.cuh"

namespace kvq {

constexpr int kBfWarps = 2;
constexpr int kBfRing = 2;
constexpr int kBfTilesPerWarp = kPart / 16 / kBfWarps;  // 16
constexpr int kBfD = 256;
constexpr int kBfRowG = kBfD * 2 + 16;  // padded row bytes of the gather layout

struct __align__(1024) BfStage {
  // dense: [4 column boxes][16 rows][128 B], 128-byte swizzled; gather: [16 rows][528 B];
  // each tile starts on a 1024-byte boundary (the swizzle pattern is address-based)
  uint8_t k[9216];
  uint8_t v[9216];
};
static_assert(16 * kBfRowG <= 9216, "gather rows fit a tile");

struct BfSmem {
  BfStage stage[kBfWarps][kBfRing];
  uint4 qf[kBfD / 16][32];  // per k-step and lane: (hi b0, hi b1, lo b0, lo b1)
  uint64_t bar[kBfWarps][kBfRing];
  int poison;
};

struct BfCombine {  // reuses the ring once every warp is done
  float acc[kBfWarps][8][kBfD];
  float m[kBfWarps][8];
  float z[kBfWarps][8];
};
static_assert(sizeof(BfCombine) <= sizeof(BfStage) * kBfWarps * kBfRing, "combine fits in the ring");
static_assert(sizeof(BfSmem) + 1024 <= 232448, "bf16 decode shared memory");

__device__ __forceinline__ void bf_tma_2d(void* dst, const CUtensorMap* map, int x, int row, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(row), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bf_ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void bf_ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint4 bf_lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// Split (x0, x1) into bf16 high and low parts: x ~= hi + lo to ~16 bits.
__device__ __forceinline__ void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Byte offset of (row r, 16-byte chunk c of the 512-byte row) in a stage's K or V tile.
template <bool GATHER>
__device__ __forceinline__ uint32_t bf_off(int r, int c) {
  if (GATHER) return r * kBfRowG + 16 * c;
  return (c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4);
}

// Issue the copies of one 16-key tile.  Returns false if a page or a selected
// index is invalid (the tile then counts as poisoned; its barrier is still
// completed so the consumer does not wait on it).
template <bool GATHER>
__device__ __forceinline__ bool bf_issue_tile(const DecodeArgs& a, int b, int kvh, int key0, int nvalid, int32_t page,
                                              BfStage* st, uint64_t* bar) {
  const kvq_cache& c = a.c;
  if constexpr (!GATHER) {
    if (page < 0 || page >= c.num_pages) {
      set_status(a.status, KVQ_DEV_BAD_PAGE);
      mbar_arrive(bar);
      return false;
    }
    const int row0 = static_cast<int>(((int64_t)page * c.num_kv_heads + kvh) * c.page_size + key0 % c.page_size);
    mbar_arrive_expect_tx(bar, 2 * 16 * kBfD * 2);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      bf_tma_2d(st->k + x * 2048, &a.tm_k, 128 * x, row0, bar);
      bf_tma_2d(st->v + x * 2048, &a.tm_v, 128 * x, row0, bar);
    }
    return true;
  } else {
    const int32_t T = a.seq_lens[b];
    const int32_t* bt = a.block_tables + (int64_t)b * a.max_pages;
    int64_t rows[16];
    for (int j = 0; j < nvalid; ++j) {
      const int32_t pos = a.sel[(int64_t)b * a.n_sel + key0 + j];
      int32_t pg = -1;
      if (pos < 0 || pos >= T) {
        set_status(a.status, KVQ_DEV_BAD_INDEX);
      } else {
        pg = bt[pos / c.page_size];
        if (pg < 0 || pg >= c.num_pages) set_status(a.status, KVQ_DEV_BAD_PAGE);
      }
      if (pg < 0 || pg >= c.num_pages) {
        mbar_arrive(bar);
        return false;
      }
      rows[j] = ((int64_t)pg * c.num_kv_heads + kvh) * c.page_size + pos % c.page_size;
    }
    mbar_arrive_expect_tx(bar, nvalid * 2 * kBfD * 2);
    for (int j = 0; j < nvalid; ++j) {
      bulk_g2s(st->k + j * kBfRowG, static_cast<const uint8_t*>(c.k) + rows[j] * (kBfD * 2), kBfD * 2, bar);
      bulk_g2s(st->v + j * kBfRowG, static_cast<const uint8_t*>(c.v) + rows[j] * (kBfD * 2), kBfD * 2, bar);
    }
    return true;
  }
}

template <bool GATHER>
__global__ void __launch_bounds__(kBfWarps * 32, 2) decode_bf16_kernel(const __grid_constant__ DecodeArgs a) {
  pdl_wait();
  extern __shared__ uint8_t smem_raw[];
  BfSmem& sm = *reinterpret_cast<BfSmem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
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
  const int my_first = warp * kBfTilesPerWarp;
  const int my_tiles = max(0, min(kBfTilesPerWarp, ntiles - my_first));

  int32_t my_page = -1;  // page of this warp's tile `lane`
  if (!GATHER && lane < my_tiles)
    my_page = a.block_tables[(int64_t)b * a.max_pages + (k0 + 16 * (my_first + lane)) / a.c.page_size];
  int32_t first_pages[kBfRing];
#pragma unroll
  for (int i = 0; i < kBfRing; ++i) first_pages[i] = __shfl_sync(0xffffffffu, my_page, i);

  bool poisoned = false;
  if (lane == 0) {
    for (int s = 0; s < kBfRing; ++s) mbar_init(&sm.bar[warp][s], 1);
    fence_barrier_init();
    for (int i = 0; i < min(kBfRing, my_tiles); ++i) {
      const int key0 = k0 + 16 * (my_first + i);
      if (!bf_issue_tile<GATHER>(a, b, kvh, key0, min(16, k1 - key0), first_pages[i], &sm.stage[warp][i],
                                 &sm.bar[warp][i]))
        poisoned = true;
    }
  }
  if (threadIdx.x == 0) sm.poison = 0;

  // ---- query fragments (B operand of the score MMA): lane (g, t) of k-step s
  // holds q[head g][16s + 2t, +1] and q[head g][16s + 2t + 8, +9], high and low.
  {
    const bool live = g < a.group;
    const float* qrow = a.q + ((int64_t)b * a.Hq + kvh * a.group + (live ? g : 0)) * kBfD;
    const float sc = live ? a.qscale : 0.f;
    constexpr int kSteps = kBfD / 16 / kBfWarps;  // k-steps per warp; all loads issued first
    float2 u0[kSteps], u1[kSteps];
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
      const int s = warp + kBfWarps * k;
      u0[k] = *reinterpret_cast<const float2*>(qrow + 16 * s + 2 * t);
      u1[k] = *reinterpret_cast<const float2*>(qrow + 16 * s + 2 * t + 8);
    }
#pragma unroll
    for (int k = 0; k < kSteps; ++k) {
      uint4 f;
      split_bf16(u0[k].x * sc, u0[k].y * sc, f.x, f.z);
      split_bf16(u1[k].x * sc, u1[k].y * sc, f.y, f.w);
      sm.qf[warp + kBfWarps * k][lane] = f;
    }
  }
  __syncthreads();
  const uint32_t qf_addr = smem_u32(&sm.qf[0][lane]);

  float acc[kBfD / 16][4];  // O^T: dims 16 mb + g (+8), heads 2t, 2t+1
#pragma unroll
  for (int mb = 0; mb < kBfD / 16; ++mb)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mb][i] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY;
  float z0 = 0.f, z1 = 0.f;
  const bool head0_live = 2 * t < a.group, head1_live = 2 * t + 1 < a.group;
  bool timed_out = false;
  // ldmatrix lane roles: K (scores): rows (lane & 7) + 8((lane >> 3) & 1), chunk + (lane >> 4);
  //                      V^T (context, .trans): rows (lane & 7) + 8(lane >> 4), chunk + ((lane >> 3) & 1)
  const int kr = (lane & 7) + 8 * ((lane >> 3) & 1), kc = lane >> 4;
  const int vr = (lane & 7) + 8 * (lane >> 4), vc = (lane >> 3) & 1;

  for (int i = 0; i < my_tiles; ++i) {
    const int s = i % kBfRing;
    BfStage& st = sm.stage[warp][s];
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sm.bar[warp][s], (i / kBfRing) & 1))) {
      timed_out = true;
      break;
    }
    const uint32_t kb = smem_u32(st.k), vb = smem_u32(st.v);
    const int key0 = k0 + 16 * (my_first + i);
    const int nvalid = min(16, k1 - key0);

    // ---------------- scores S[key][head] for keys g, g+8 and heads 2t, 2t+1
    float Sh[4] = {0.f, 0.f, 0.f, 0.f}, Sl[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ks = 0; ks < kBfD / 16; ++ks) {
      uint32_t ak[4];
      bf_ldsm_x4(kb + bf_off<GATHER>(kr, 2 * ks + kc), ak);
      const uint4 q = bf_lds128(qf_addr + ks * 512);
      mma_bf16(Sh, ak[0], ak[1], ak[2], ak[3], q.x, q.y);
      mma_bf16(Sl, ak[0], ak[1], ak[2], ak[3], q.z, q.w);
    }
    float S[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) S[j] = Sh[j] + Sl[j];
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
    if (i > 0 && __any_sync(0xffffffffu, c0 != 1.f || c1 != 1.f)) {
#pragma unroll
      for (int mb = 0; mb < kBfD / 16; ++mb) {
        acc[mb][0] *= c0;
        acc[mb][1] *= c1;
        acc[mb][2] *= c0;
        acc[mb][3] *= c1;
      }
    }

    // ---------------- P (keys x heads) -> B fragments, bf16 high and low parts
    uint32_t ph01, pl01, ph23, pl23;
    split_bf16(p0, p1, ph01, pl01);
    split_bf16(p2, p3, ph23, pl23);
    const uint32_t bh0 = movmatrix_trans(ph01), bl0 = movmatrix_trans(pl01);  // keys 2t, 2t+1 of head g
    const uint32_t bh1 = movmatrix_trans(ph23), bl1 = movmatrix_trans(pl23);  // keys 2t+8, 2t+9
    // V rows past the end hold stale or unwritten bytes; their P is 0, but 0 x NaN
    // would still poison the sum, so those rows are zeroed first (tail tile only).
    if (nvalid < 16) {
      for (int r = nvalid; r < 16; ++r)  // lane = 16-byte chunk of the 512-byte row
        *reinterpret_cast<uint4*>(&st.v[bf_off<GATHER>(r, lane)]) = make_uint4(0, 0, 0, 0);
      fence_proxy_async();  // before the stage is refilled by the copy engine
      __syncwarp();
    }

    // ---------------- context: O^T[dims][heads] += V^T . P^T
#pragma unroll
    for (int mb = 0; mb < kBfD / 16; ++mb) {
      uint32_t av[4];
      bf_ldsm_x4_t(vb + bf_off<GATHER>(vr, 2 * mb + vc), av);
      mma_bf16(acc[mb], av[0], av[1], av[2], av[3], bh0, bh1);
      mma_bf16(acc[mb], av[0], av[1], av[2], av[3], bl0, bl1);
    }

    const int32_t next_page = __shfl_sync(0xffffffffu, my_page, min(i + kBfRing, 31));
    __syncwarp();
    if (lane == 0 && i + kBfRing < my_tiles) {
      fence_proxy_async();
      const int nk0 = k0 + 16 * (my_first + i + kBfRing);
      if (!bf_issue_tile<GATHER>(a, b, kvh, nk0, min(16, k1 - nk0), next_page, &st, &sm.bar[warp][s]))
        poisoned = true;
    }
  }
  if (timed_out && lane == 0) set_status(a.status, KVQ_DEV_TIMEOUT);
  poisoned = __any_sync(0xffffffffu, poisoned || timed_out);

#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    z0 += __shfl_xor_sync(0xffffffffu, z0, o);
    z1 += __shfl_xor_sync(0xffffffffu, z1, o);
  }
  if (poisoned && lane == 0) atomicOr(&sm.poison, 1);
  __syncthreads();  // every warp is done with the ring
  BfCombine& cb = *reinterpret_cast<BfCombine*>(&sm.stage[0][0]);
#pragma unroll
  for (int mb = 0; mb < kBfD / 16; ++mb) {
    cb.acc[warp][2 * t][16 * mb + g] = acc[mb][0];
    cb.acc[warp][2 * t + 1][16 * mb + g] = acc[mb][1];
    cb.acc[warp][2 * t][16 * mb + g + 8] = acc[mb][2];
    cb.acc[warp][2 * t + 1][16 * mb + g + 8] = acc[mb][3];
  }
  if (g == 0) {
    cb.m[warp][2 * t] = m0;
    cb.m[warp][2 * t + 1] = m1;
    cb.z[warp][2 * t] = z0;
    cb.z[warp][2 * t + 1] = z1;
  }
  __syncthreads();
  const bool bad = sm.poison != 0;
  for (int idx = threadIdx.x; idx < a.group * (kBfD / 4); idx += blockDim.x) {
    const int h = idx / (kBfD / 4), d4 = idx % (kBfD / 4);
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kBfWarps; ++w) M = fmaxf(M, cb.m[w][h]);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float Z = 0.f;
#pragma unroll
    for (int w = 0; w < kBfWarps; ++w) {
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
    *reinterpret_cast<float4*>(a.ws_acc + pi * kBfD + 4 * d4) = o;
    if (d4 == 0) {
      a.ws_m[pi] = bad ? NAN : M;
      a.ws_z[pi] = bad ? NAN : Z;
    }
  }
  pdl_trigger();  // after this CTA's last write
}

cudaError_t launch_decode_bf16(const DecodeArgs& a, int B, cudaStream_t s) {
  const size_t smem = sizeof(BfSmem) + 1024;
  dim3 grid(a.P, a.c.num_kv_heads, B);
  if (a.sel) {
    cudaError_t e = set_max_smem_once<decode_bf16_kernel<true>>((int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_bf16_kernel<true>, grid, dim3(kBfWarps * 32), smem, s, a);
    if (e != cudaSuccess) return e;
  } else {
    cudaError_t e = set_max_smem_once<decode_bf16_kernel<false>>((int)smem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(decode_bf16_kernel<false>, grid, dim3(kBfWarps * 32), smem, s, a);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace kvq
