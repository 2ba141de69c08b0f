// prefill_q4.cu -- causal attention of a prompt chunk over the decoded 4-bit slots.
//
// Follows "qwen27 CUDA: an opt-in 4-bit attention cache (262K on a 24 GB card)",
// section "What it is": prompt chunks are packed into the cache and attended
// with the prefill-attention kernel over decoded slots.  Query i of the chunk
// sits at absolute position q_start + i and attends keys 0 .. q_start + i.
//
// CUDA-core kernel: one CTA (256 threads) per (query row, KV head).  The GQA
// group's queries are rotated in shared memory (warp-level FWHT), keys and
// values are decoded 32 rows at a time into shared memory in the rotated space,
// a warp per key forms the scores of the group, the online softmax runs per
// head, one thread per value element accumulates the context, and the result is
// rotated back.
#include "kernels.cuh"

namespace kvq {

constexpr int kPfChunk = 32;
constexpr int kPfD = 256;

__device__ __forceinline__ float q4_value(const uint8_t* row, const uint16_t* sc, int e) {
  const int G = e >> 5, i = e & 31;
  const int h = i >> 2, j = i & 3;
  const uint8_t byte = row[2 * (h * 8 + G) + (j >> 1)];
  const int code = (j & 1) ? (byte >> 4) : (byte & 0xF);
  return static_cast<float>(code - 8) * __half2float(__ushort_as_half(sc[G]));
}

__global__ void __launch_bounds__(256) prefill_q4_simple_kernel(const PrefillArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;                      // [8][D]
  float* ks = qs + 8 * kPfD;           // [chunk][D]
  float* vs = ks + kPfChunk * kPfD;    // [chunk][D]
  float* ps = vs + kPfChunk * kPfD;    // [8][chunk]
  float* mz = ps + 8 * kPfChunk;       // m[8], z[8], corr[8]
  __shared__ int s_bad;
  const int qi = blockIdx.x, kvh = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const kvq_cache& c = a.c;
  const int nh = a.group;
  const int T = a.q_start + qi + 1;

  // rotated queries of the group, pre-scaled
  for (int task = warp; task < 8 * (kPfD / 32); task += 8) {
    const int h = task / (kPfD / 32), G = task % (kPfD / 32);
    float x = 0.f;
    if (h < nh) {
      const int64_t idx = ((int64_t)qi * a.Hq + kvh * a.group + h) * kPfD + 32 * G + lane;
      x = a.dtype == KVQ_DT_F32 ? static_cast<const float*>(a.q)[idx]
                                : __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[idx]);
      x = __fmul_rn(warp_fwht32(x, lane), kHadamardScale) * a.qscale;
    }
    qs[h * kPfD + 32 * G + lane] = x;
  }
  if (tid < 8) {
    mz[tid] = -INFINITY;
    mz[8 + tid] = 0.f;
  }
  if (tid == 0) s_bad = 0;
  float acc[8];
#pragma unroll
  for (int h = 0; h < 8; ++h) acc[h] = 0.f;
  __syncthreads();

  for (int kc = 0; kc < T; kc += kPfChunk) {
    const int nk = min(kPfChunk, T - kc);
    for (int j = warp; j < kPfChunk; j += 8) {
      bool ok = j < nk;
      int64_t r = 0;
      if (ok) {
        const int pos = kc + j;
        const int32_t page = a.block_table[pos / c.page_size];
        if (page < 0 || page >= c.num_pages) {
          if (lane == 0) { set_status(a.status, KVQ_DEV_BAD_PAGE); s_bad = 1; }
          ok = false;
        } else {
          r = ((int64_t)page * c.num_kv_heads + kvh) * c.page_size + pos % c.page_size;
        }
      }
      const uint8_t* kr = static_cast<const uint8_t*>(c.k) + r * (kPfD / 2);
      const uint8_t* vr = static_cast<const uint8_t*>(c.v) + r * (kPfD / 2);
      const uint16_t* ksc = static_cast<const uint16_t*>(c.k_scale) + r * (kPfD / 32);
      const uint16_t* vsc = static_cast<const uint16_t*>(c.v_scale) + r * (kPfD / 32);
      for (int e = lane; e < kPfD; e += 32) {
        ks[j * kPfD + e] = ok ? q4_value(kr, ksc, e) : 0.f;
        vs[j * kPfD + e] = ok ? q4_value(vr, vsc, e) : 0.f;
      }
    }
    __syncthreads();
    for (int j = warp; j < nk; j += 8) {
      float part[8];
#pragma unroll
      for (int h = 0; h < 8; ++h) part[h] = 0.f;
      for (int d = lane; d < kPfD; d += 32) {
        const float kv = ks[j * kPfD + d];
#pragma unroll
        for (int h = 0; h < 8; ++h) part[h] = fmaf(qs[h * kPfD + d], kv, part[h]);
      }
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        float v = part[h];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) ps[h * kPfChunk + j] = v;
      }
    }
    __syncthreads();
    {
      const int h = warp;
      if (h < nh) {
        const float s = lane < nk ? ps[h * kPfChunk + lane] : -INFINITY;
        float tm = s;
        for (int o = 16; o > 0; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
        const float mo = mz[h], mn = fmaxf(mo, tm);
        const float pr = lane < nk ? exp2f(s - mn) : 0.f;
        float sum = pr;
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        ps[h * kPfChunk + lane] = pr;
        __syncwarp();
        if (lane == 0) {
          const float corr = exp2f(mo - mn);
          mz[h] = mn;
          mz[8 + h] = mz[8 + h] * corr + sum;
          mz[16 + h] = corr;
        }
      } else if (lane == 0) {
        mz[16 + h] = 1.f;
      }
    }
    __syncthreads();
    const int d = tid;
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      float o = acc[h] * mz[16 + h];
      for (int j = 0; j < nk; ++j) o = fmaf(ps[h * kPfChunk + j], vs[j * kPfD + d], o);
      acc[h] = o;
    }
    __syncthreads();
  }
  // normalise, rotate back (warp per group via shared memory), store
  const bool bad = s_bad != 0;
#pragma unroll
  for (int h = 0; h < 8; ++h) ks[h * kPfD + tid] = (h < nh) ? acc[h] / mz[8 + h] : 0.f;
  __syncthreads();
  for (int task = warp; task < nh * (kPfD / 32); task += 8) {
    const int h = task / (kPfD / 32), G = task % (kPfD / 32);
    float x = ks[h * kPfD + 32 * G + lane];
    x = __fmul_rn(warp_fwht32(x, lane), kHadamardScale);
    a.out[((int64_t)qi * a.Hq + kvh * a.group + h) * kPfD + 32 * G + lane] = bad ? NAN : x;
  }
}

cudaError_t launch_prefill_q4(const PrefillArgs& a, cudaStream_t s) {
  if (a.n_q == 0) return cudaSuccess;
  const size_t smem = sizeof(float) * (8 * kPfD + 2 * kPfChunk * kPfD + 8 * kPfChunk + 24);
  cudaError_t e = cudaFuncSetAttribute(prefill_q4_simple_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_q, a.c.num_kv_heads);
  prefill_q4_simple_kernel<<<grid, 256, smem, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
