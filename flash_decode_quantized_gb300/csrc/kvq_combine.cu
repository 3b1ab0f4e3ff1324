// Split-K combine (step a8): merges the per-chunk partials (m, l, acc) of every query head.
//
// With chunk partials m_c (running max of the base-2 logits), l_c = sum 2^(s - m_c) and
// acc_c = sum 2^(s - m_c) v, the output is
//   out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c,  M = max_c m_c,
// the flash-decode reduction of the split over kv_len.  Every sum runs in a fixed order
// (chunk index, then a fixed tree), so the result does not depend on which CTA of the
// decode kernel finished first.
//
// One CTA per (query head, sequence): its threads split the chunks, and each thread owns
// one element of head_dim in the weighted sum (loads of a chunk's partial row coalesce).
// The kernel is launched with programmatic stream serialization, so its launch overlaps
// the tail of the decode kernel; griddepcontrol.wait orders it after that kernel's writes.
#include "kvq_device.cuh"

namespace kvq {

namespace {

constexpr int kCombineThreads = 256;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < kCombineThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  return r;
}

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(DecodeArgs a, int D) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ float red[kCombineThreads / 32];
  __shared__ float part[kCombineThreads];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const long long cap = min((long long)a.max_pages * a.k.page_size, (long long)a.n_chunks * a.chunk_tokens);
  long long L = a.seq_lens[b];
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int nv = (int)((L + a.chunk_tokens - 1) / a.chunk_tokens);
  const long long head = (long long)b * a.num_q_heads + h;
  const float* ml = a.part_ml + head * a.n_chunks * 2;
  const float* po = a.part_o + head * a.n_chunks * D;

  float M = -INFINITY;
  for (int c = tid; c < nv; c += kCombineThreads) M = fmaxf(M, ml[2 * c]);
  M = block_reduce(M, true, red);
  float den = 0.0f;
  for (int c = tid; c < nv; c += kCombineThreads)
    if (ml[2 * c] != -INFINITY) den += fast_exp2(ml[2 * c] - M) * ml[2 * c + 1];
  den = block_reduce(den, false, red);

  // thread (j, g): element j, chunks g, g + groups, ...
  const int groups = kCombineThreads / D;
  const int j = tid % D, g = tid / D;
  float num = 0.0f;
  if (g < groups) {
    int c = g;
    for (; c + 3 * groups < nv; c += 4 * groups) {
      float w[4], v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float m = ml[2 * (c + u * groups)];
        w[u] = (m == -INFINITY) ? 0.0f : fast_exp2(m - M);
        v[u] = po[(long long)(c + u * groups) * D + j];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) num = fmaf(w[u], v[u], num);
    }
    for (; c < nv; c += groups) {
      const float m = ml[2 * c];
      if (m != -INFINITY) num = fmaf(fast_exp2(m - M), po[(long long)c * D + j], num);
    }
  }
  part[tid] = num;
  __syncthreads();
  if (tid < D) {
    float s = 0.0f;
    for (int gg = 0; gg < groups; ++gg) s += part[gg * D + tid];
    a.out[head * D + tid] = den > 0.0f ? s / den : 0.0f;
  }
}

}  // namespace

cudaError_t launch_combine_pdl(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_q_heads, a.batch);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel, a, head_dim);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace kvq
