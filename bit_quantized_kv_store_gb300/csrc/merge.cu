// merge.cu -- log-sum-exp merge of split-T partials, then the rotation back.
//
// Follows "qwen27 CUDA: an opt-in 4-bit attention cache (262K on a 24 GB card)",
// section "What it is" (an in-order merge, then rotate the output back once) and
// "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", split-T commit (a
// log-sum-exp merge kernel over the (m, z, cl) partials).
//
// One CTA of 256 threads per (32 output values, query head, sequence).  The
// partitions are read as float4 rows; thread i takes partitions i/8, i/8 + 32,
// ... in ascending order, and the 32 per-thread sums are then added in a fixed
// tree, so the result does not depend on scheduling (bit-reproducible).  The
// 32 values of a CTA are exactly one Hadamard group, rotated back in one warp.
#include "kernels.cuh"

namespace kvq {

__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs a) {
  pdl_wait();
  pdl_trigger();
  const int grp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float* outp = a.out + ((int64_t)b * a.Hq + h) * a.Dv + 32 * grp;
  int32_t T;
  bool bad = false;
  if (a.n_sel > 0) {
    T = a.n_sel;
  } else {
    T = a.seq_lens[b];
    bad = T < 0 || T > a.max_seq_len;
  }
  if (bad) {
    if (tid < 32) outp[tid] = NAN;
    return;
  }
  const int np = (T + kPart - 1) / kPart;
  if (np == 0) {
    if (tid < 32) outp[tid] = 0.f;
    return;
  }
  const int64_t base = ((int64_t)b * a.Hq + h) * a.P;
  const float* m = a.ws_m + base;
  const float* z = a.ws_z + base;

  __shared__ float red[8];
  __shared__ float red_acc[32][33];
  __shared__ float s_M, s_Z;
  __shared__ int s_nan;

  // M = max_p m_p (NaN anywhere poisons the result)
  float mx = -INFINITY;
  int nan_seen = 0;
  for (int i = tid; i < np; i += 256) {
    const float v = m[i];
    nan_seen |= isnan(v);
    mx = fmaxf(mx, v);
  }
  for (int o = 16; o > 0; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    nan_seen |= __shfl_xor_sync(0xffffffffu, nan_seen, o);
  }
  if (tid == 0) s_nan = 0;
  __syncthreads();
  if (lane == 0) {
    red[warp] = mx;
    if (nan_seen) s_nan = 1;
  }
  __syncthreads();
  if (tid == 0) {
    float M = red[0];
    for (int w = 1; w < 8; ++w) M = fmaxf(M, red[w]);
    s_M = M;
  }
  __syncthreads();
  const float M = s_M;
  const bool empty = (M == -INFINITY);

  // Z = sum_p z_p 2^(m_p - M), per-thread ascending, then a fixed tree
  float zs = 0.f;
  for (int i = tid; i < np; i += 256) zs += empty ? 0.f : z[i] * exp2f(m[i] - M);
  for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);
  __syncthreads();
  if (lane == 0) red[warp] = zs;
  __syncthreads();
  if (tid == 0) {
    float Z = 0.f;
    for (int w = 0; w < 8; ++w) Z += red[w];
    s_Z = Z;
  }

  // acc: thread covers float4 chunk (tid % 8) of the group, partitions tid/8 + 32k
  const int chunk = tid & 7, prow = tid >> 3;
  float4 s4 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!empty) {
    for (int i = prow; i < np; i += 32) {
      const float w = exp2f(m[i] - M);
      const float4 v = *reinterpret_cast<const float4*>(a.ws_acc + (base + i) * a.Dv + 32 * grp + 4 * chunk);
      s4.x = fmaf(v.x, w, s4.x);
      s4.y = fmaf(v.y, w, s4.y);
      s4.z = fmaf(v.z, w, s4.z);
      s4.w = fmaf(v.w, w, s4.w);
    }
  }
  red_acc[prow][4 * chunk + 0] = s4.x;
  red_acc[prow][4 * chunk + 1] = s4.y;
  red_acc[prow][4 * chunk + 2] = s4.z;
  red_acc[prow][4 * chunk + 3] = s4.w;
  __syncthreads();
  if (warp == 0) {
    float o = 0.f;
    for (int r = 0; r < 32; ++r) o += red_acc[r][lane];  // ascending partition rows
    const float Z = s_Z;
    o = (empty || Z == 0.f) ? 0.f : o / Z;
    if (s_nan) o = NAN;
    if (a.rotate_back) o = __fmul_rn(warp_fwht32(o, lane), kHadamardScale);
    outp[lane] = o;
  }
}

cudaError_t launch_merge(const MergeArgs& a, int B, cudaStream_t s) {
  dim3 grid(a.Dv / 32, a.Hq, B);
  if (B == 0 || a.Hq == 0) return cudaSuccess;
  cudaError_t e = launch_pdl(merge_kernel, grid, dim3(256), 0, s, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvq
