// decode_rows.cu -- split-T decode partials for the row formats without
// sub-byte packing: the unrotated bf16 comparison cache and the fp8 e4m3 latent
// rows of absorbed MLA attention.
//
// fp8 rows follow "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", KV8 base
// commit (score and context loops dequantise through e4m3 with the row scale
// hoisted out of the dot; the latent is both key and value) and the split-T
// commit ((H, P) partials (cl, m, z) merged by log-sum-exp; the selected-row
// gather splits into the same partials).
//
// CUDA-core kernel: one CTA (256 threads) per (partition of 512 keys, block of
// heads, sequence).  Keys are staged in shared memory 32 at a time; a warp per
// key computes the dot products of all heads of the block (lanes split the key
// width, then a shuffle reduction); the online softmax runs per head; the
// context accumulates with one thread per value element.
#include <cuda_fp8.h>

#include "kernels.cuh"

namespace kvq {

constexpr int kRowsChunk = 32;

// FMT 1: bf16 rows of D (W = Dv = D).  FMT 2: fp8 latent D + rope R (W = D + R, Dv = D).
template <int FMT, int HB, int W, int DV>
__global__ void __launch_bounds__(256) decode_rows_kernel(const RowsArgs a) {
  extern __shared__ __align__(16) float sm[];
  float* qs = sm;                              // [HB][W]
  float* ks = qs + HB * W;                     // [chunk][W]  (fp32 values incl. scale)
  float* vs = ks + kRowsChunk * W;             // [chunk][DV]
  float* ps = vs + kRowsChunk * DV;            // [HB][chunk]
  float* mz = ps + HB * kRowsChunk;            // m[HB], z[HB], corr[HB]
  __shared__ int s_bad;

  const int p = blockIdx.x, hblk = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const kvq_cache& c = a.c;
  const int head0 = hblk * a.hb;  // first query head of this CTA (a.hb <= HB)
  const int kvh = head0 / a.group;
  const int nh = min(a.hb, a.Hq - head0);

  int32_t T;
  if (a.sel) {
    T = a.n_sel;
  } else {
    T = a.seq_lens[b];
    if (T < 0 || T > a.max_seq_len || (int64_t)T > (int64_t)a.max_pages * c.page_size) {
      if (tid == 0 && p == 0 && hblk == 0) set_status(a.status, KVQ_DEV_BAD_LENGTH);
      return;
    }
  }
  const int nparts = (T + kPart - 1) / kPart;
  if (p >= nparts) return;
  const int k0 = p * kPart, k1 = min(k0 + kPart, T);

  for (int i = tid; i < HB * W; i += 256) {
    const int h = i / W, d = i % W;
    qs[i] = h < nh ? a.q[((int64_t)b * a.Hq + head0 + h) * W + d] * a.qscale : 0.f;
  }
  if (tid < HB) {
    mz[tid] = -INFINITY;
    mz[HB + tid] = 0.f;
  }
  if (tid == 0) s_bad = 0;
  float acc[HB][DV / 256];
#pragma unroll
  for (int h = 0; h < HB; ++h)
#pragma unroll
    for (int j = 0; j < DV / 256; ++j) acc[h][j] = 0.f;
  __syncthreads();

  const int32_t* bt = a.block_tables + (int64_t)b * a.max_pages;
  const int32_t Tseq = a.seq_lens[b];
  for (int kc = k0; kc < k1; kc += kRowsChunk) {
    const int nk = min(kRowsChunk, k1 - kc);
    // ---- stage keys/values of the chunk as fp32 (value incl. row scale)
    for (int j = warp; j < kRowsChunk; j += 8) {
      bool ok = j < nk;
      int64_t r = 0;
      if (ok) {
        int32_t pos = kc + j;
        if (a.sel) {
          pos = a.sel[(int64_t)b * a.n_sel + kc + j];
          if (pos < 0 || pos >= Tseq) {
            if (lane == 0) { set_status(a.status, KVQ_DEV_BAD_INDEX); s_bad = 1; }
            ok = false;
          }
        }
        if (ok) {
          const int32_t page = bt[pos / c.page_size];
          if (page < 0 || page >= c.num_pages) {
            if (lane == 0) { set_status(a.status, KVQ_DEV_BAD_PAGE); s_bad = 1; }
            ok = false;
          } else {
            r = ((int64_t)page * c.num_kv_heads + kvh) * c.page_size + pos % c.page_size;
          }
        }
      }
      if (FMT == 1) {
        const __nv_bfloat16* kr = static_cast<const __nv_bfloat16*>(c.k) + r * W;
        const __nv_bfloat16* vr = static_cast<const __nv_bfloat16*>(c.v) + r * W;
        for (int d = lane; d < W; d += 32) {
          ks[j * W + d] = ok ? __bfloat162float(kr[d]) : 0.f;
          vs[j * DV + d] = ok ? __bfloat162float(vr[d]) : 0.f;
        }
      } else {
        constexpr int R = W - DV;
        const uint8_t* lr = static_cast<const uint8_t*>(c.k) + r * DV;
        const uint8_t* rr = static_cast<const uint8_t*>(c.v) + r * R;
        const float ls = ok ? static_cast<const float*>(c.k_scale)[r] : 0.f;
        const float rs = ok ? static_cast<const float*>(c.v_scale)[r] : 0.f;
        for (int d = lane; d < W; d += 32) {
          float x = 0.f;
          if (ok) {
            const uint8_t code = d < DV ? lr[d] : rr[d - DV];
            __nv_fp8_e4m3 f;
            f.__x = code;
            x = static_cast<float>(f) * (d < DV ? ls : rs);
          }
          ks[j * W + d] = x;
          if (d < DV) vs[j * DV + d] = x;
        }
      }
    }
    __syncthreads();
    // ---- scores: warp per key, lanes split the width
    for (int j = warp; j < nk; j += 8) {
      float part[HB];
#pragma unroll
      for (int h = 0; h < HB; ++h) part[h] = 0.f;
      for (int d = lane; d < W; d += 32) {
        const float kv = ks[j * W + d];
#pragma unroll
        for (int h = 0; h < HB; ++h) part[h] = fmaf(qs[h * W + d], kv, part[h]);
      }
#pragma unroll
      for (int h = 0; h < HB; ++h) {
        float v = part[h];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) ps[h * kRowsChunk + j] = v;
      }
    }
    __syncthreads();
    // ---- online softmax per head (base 2)
    for (int h = warp; h < HB; h += 8) {
      if (h >= nh) {
        if (lane == 0) mz[2 * HB + h] = 1.f;
        continue;
      }
      const float s = lane < nk ? ps[h * kRowsChunk + lane] : -INFINITY;
      float tm = s;
      for (int o = 16; o > 0; o >>= 1) tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, o));
      const float mo = mz[h];
      const float mn = fmaxf(mo, tm);
      const float pr = lane < nk ? exp2f(s - mn) : 0.f;
      float sum = pr;
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      ps[h * kRowsChunk + lane] = pr;
      __syncwarp();
      if (lane == 0) {
        const float corr = exp2f(mo - mn);
        mz[h] = mn;
        mz[HB + h] = mz[HB + h] * corr + sum;
        mz[2 * HB + h] = corr;
      }
    }
    __syncthreads();
    // ---- context: one thread per value element
#pragma unroll
    for (int jj = 0; jj < DV / 256; ++jj) {
      const int d = tid + 256 * jj;
#pragma unroll
      for (int h = 0; h < HB; ++h) {
        float o = acc[h][jj] * mz[2 * HB + h];
        for (int j = 0; j < nk; ++j) o = fmaf(ps[h * kRowsChunk + j], vs[j * DV + d], o);
        acc[h][jj] = o;
      }
    }
    __syncthreads();
  }
  const bool bad = s_bad != 0;
#pragma unroll
  for (int h = 0; h < HB; ++h) {
    if (h >= nh) break;
    const int64_t pi = ((int64_t)b * a.Hq + head0 + h) * a.P + p;
#pragma unroll
    for (int jj = 0; jj < DV / 256; ++jj) a.ws_acc[pi * DV + tid + 256 * jj] = bad ? NAN : acc[h][jj];
    if (tid == 0) {
      a.ws_m[pi] = bad ? NAN : mz[h];
      a.ws_z[pi] = bad ? NAN : mz[HB + h];
    }
  }
}

template <int FMT, int HB, int W, int DV>
static cudaError_t launch_rows_t(const RowsArgs& a, int B, cudaStream_t s) {
  const size_t smem = sizeof(float) * (HB * W + kRowsChunk * W + kRowsChunk * DV + HB * kRowsChunk + 3 * HB);
  cudaError_t e = cudaFuncSetAttribute(decode_rows_kernel<FMT, HB, W, DV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.P, (a.Hq + a.hb - 1) / a.hb, B);
  decode_rows_kernel<FMT, HB, W, DV><<<grid, 256, smem, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_decode_rows(const RowsArgs& a, int B, cudaStream_t s) {
  if (a.c.format == KVQ_FMT_BF16) {
    // one CTA per KV head: the GQA group shares each staged key
    return launch_rows_t<1, 8, 256, 256>(a, B, s);
  }
  return launch_rows_t<2, 16, 576, 512>(a, B, s);
}

}  // namespace kvq
