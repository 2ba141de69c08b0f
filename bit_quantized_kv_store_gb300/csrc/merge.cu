// merge.cu -- log-sum-exp merge of split-T partials, then the rotation back.
//
// Follows "qwen27 CUDA: an opt-in 4-bit attention cache (262K on a 24 GB card)",
// section "What it is" (an in-order merge, then rotate the output back once) and
// "KV cache quantization: fp8 (KV8) + 4-bit TurboQuant", split-T commit (a
// log-sum-exp merge kernel over the (m, z, cl) partials).
//
// One CTA of 256 threads per (32 output values, query head, sequence), one
// pass over the partials.  Thread (row r = tid / 8, chunk c = tid % 8) takes
// partitions r, r + 32, r + 64, ... in ascending order: it loads their m (and,
// for c == 0, z) and the float4 chunk c of their acc, four (or eight)
// partitions per batch with every load of a batch issued before any use, and keeps a running
// (M_t, Z_t, acc_t) rescaled to its own maximum.  The 32 row-threads' partials
// are then combined in a fixed tree, so the result does not depend on
// scheduling (bit-reproducible), and the 32 values of the CTA -- exactly one
// Hadamard group -- are rotated back in one warp.  (The TQ4 rows' transform
// spans the whole row, so their rotation back is a second launch, tq4.cu.)
// The number of keys per partition comes with the arguments: 512, or for the
// fp8 streaming prefill one partition per row, whose length is q_start + row + 1.
#include "kernels.cuh"

namespace kvq {

// kBatch: partitions a row-thread loads before using them (4; for a grid of few
// CTAs over many partitions 8, or 17 past 256 partitions, so that a 262K-key
// sequence's 513 take one round trip, still at two CTAs per SM: fewer round
// trips, more registers; for a grid of many waves 2, at six CTAs per SM: more
// CTAs resident, more round trips); the updates run in ascending partition
// order either way, so the bits are the same.
template <int kBatch>
__global__ void __launch_bounds__(256, kBatch > 8 ? 2 : kBatch == 2 ? 6 : 1) merge_kernel(const MergeArgs a) {
  pdl_wait();
  pdl_trigger();
  const int grp = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31;
  float* outp = a.out + ((int64_t)b * a.Hq + h) * a.Dv + 32 * grp;
  int32_t T;
  bool bad = false;
  if (a.n_sel > 0) {
    T = a.n_sel;
  } else {
    T = a.prefill ? a.prefill_q0 + b + 1 : a.seq_lens[b];
    bad = T < 0 || T > a.max_seq_len;
  }
  if (bad) {
    if (tid < 32) outp[tid] = NAN;
    return;
  }
  const int np = static_cast<int>(((int64_t)T + a.part - 1) / a.part);
  if (np == 0) {
    if (tid < 32) outp[tid] = 0.f;
    return;
  }
  const int64_t base = ((int64_t)b * a.Hq + h) * a.P;
  const float* m = a.ws_m + base;
  const float* z = a.ws_z + base;
  const int chunk = tid & 7, row = tid >> 3;
  const float* accp = a.ws_acc + base * a.Dv + 32 * grp + 4 * chunk;

  __shared__ float s_m[32], s_z[32];  // per row: its maximum, then its z rescaled to the CTA's
  __shared__ float red_acc[32][33];
  __shared__ int s_nan;
  if (tid == 0) s_nan = 0;

  // per-thread running partial over partitions row, row + 32, ...
  float Mt = -INFINITY, Zt = 0.f;
  float4 At = make_float4(0.f, 0.f, 0.f, 0.f);
  int nan_seen = 0;
  for (int i0 = row; i0 < np; i0 += kBatch * 32) {
    float mv[kBatch], zv[kBatch];
    float4 av[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {  // all loads of the batch first
      const int i = i0 + 32 * k;
      mv[k] = -INFINITY;
      zv[k] = 0.f;
      av[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (i < np) {
        mv[k] = m[i];
        if (chunk == 0) zv[k] = z[i];
        av[k] = *reinterpret_cast<const float4*>(accp + (int64_t)i * a.Dv);
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      if (i0 + 32 * k >= np) break;
      nan_seen |= isnan(mv[k]);
      const float Mn = fmaxf(Mt, mv[k]);
      if (Mn == -INFINITY) continue;  // nothing attended so far
      const float wo = exp2f(Mt - Mn), wn = exp2f(mv[k] - Mn);
      Zt = fmaf(Zt, wo, zv[k] * wn);
      At.x = fmaf(At.x, wo, av[k].x * wn);
      At.y = fmaf(At.y, wo, av[k].y * wn);
      At.z = fmaf(At.z, wo, av[k].z * wn);
      At.w = fmaf(At.w, wo, av[k].w * wn);
      Mt = Mn;
    }
  }
  nan_seen = __any_sync(0xffffffffu, nan_seen);
  __syncthreads();  // s_nan initialised
  if (nan_seen && lane == 0) s_nan = 1;
  if (chunk == 0) {
    s_m[row] = Mt;
    s_z[row] = Zt;
  }
  __syncthreads();
  // M = max over the 32 rows; each row's partial rescaled to M
  float M = s_m[0];
#pragma unroll
  for (int r = 1; r < 32; ++r) M = fmaxf(M, s_m[r]);
  const bool empty = (M == -INFINITY);
  const float wr = (empty || Mt == -INFINITY) ? 0.f : exp2f(Mt - M);
  red_acc[row][4 * chunk + 0] = At.x * wr;
  red_acc[row][4 * chunk + 1] = At.y * wr;
  red_acc[row][4 * chunk + 2] = At.z * wr;
  red_acc[row][4 * chunk + 3] = At.w * wr;
  __syncthreads();  // every thread has read s_m
  if (chunk == 0) s_z[row] = Zt * wr;
  __syncthreads();
  if (tid < 32) {
    float o = 0.f, Z = 0.f;
#pragma unroll
    for (int r = 0; r < 32; ++r) {  // ascending rows, a fixed order (unrolled: the loads go ahead of the adds)
      o += red_acc[r][lane];
      Z += s_z[r];
    }
    o = (empty || Z == 0.f) ? 0.f : o / Z;
    if (s_nan) o = NAN;
    if (a.rotate_back) o = __fmul_rn(warp_fwht32(o, lane), kHadamardScale);
    outp[lane] = o;
  }
}

// One thread waits, with the bounded wait of the copy waits, on a barrier that
// expects one arrival that never comes; it records the timeout and returns.
__global__ void wait_timeout_probe_kernel(int32_t* status) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (!mbar_wait_bounded(&bar, 0)) set_status(status, KVQ_DEV_TIMEOUT);
}

cudaError_t launch_wait_timeout_probe(int32_t* status, cudaStream_t s) {
  wait_timeout_probe_kernel<<<1, 1, 0, s>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, int B, cudaStream_t s) {
  dim3 grid(a.Dv / 32, a.Hq, B);
  if (B == 0 || a.Hq == 0) return cudaSuccess;
  const int64_t ctas = (int64_t)grid.x * grid.y * grid.z;
  const int64_t n_sm = device_sm_count();
  const bool deep = a.P > 128 && ctas <= 2 * n_sm;
  const bool wide = ctas > 8 * n_sm;  // many waves: more CTAs resident per SM
  cudaError_t e = deep ? (a.P > 256 ? launch_pdl(merge_kernel<17>, grid, dim3(256), 0, s, a)
                                    : launch_pdl(merge_kernel<8>, grid, dim3(256), 0, s, a))
                       : wide ? launch_pdl(merge_kernel<2>, grid, dim3(256), 0, s, a)
                              : launch_pdl(merge_kernel<4>, grid, dim3(256), 0, s, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace kvq
