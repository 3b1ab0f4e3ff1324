// Split-K combine (step a8): merges the per-chunk partials (m, l, acc) of every query head.
//
// With chunk partials m_c (running max of the base-2 logits), l_c = sum 2^(s - m_c) and
// acc_c = sum 2^(s - m_c) v, the output is
//   out = sum_c 2^(m_c - M) acc_c / sum_c 2^(m_c - M) l_c,  M = max_c m_c,
// the flash-decode reduction of the split over kv_len.  Chunks are read in index order,
// so the result does not depend on which CTA finished first.
#include "kvq_device.cuh"

namespace kvq {

namespace {

__global__ void combine_kernel(DecodeArgs a, int D) {
  const int h = blockIdx.x, b = blockIdx.y;
  const long long cap = min((long long)a.max_pages * a.k.page_size, (long long)a.n_chunks * a.chunk_tokens);
  long long L = a.seq_lens[b];
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int nv = (int)((L + a.chunk_tokens - 1) / a.chunk_tokens);
  const long long head = (long long)b * a.num_q_heads + h;
  const float* ml = a.part_ml + head * a.n_chunks * 2;
  const float* po = a.part_o + head * a.n_chunks * D;
  float M = -INFINITY;
  for (int c = 0; c < nv; ++c) M = fmaxf(M, ml[2 * c]);
  float den = 0.0f;
  for (int c = 0; c < nv; ++c)
    if (ml[2 * c] != -INFINITY) den += fast_exp2(ml[2 * c] - M) * ml[2 * c + 1];
  for (int j = threadIdx.x; j < D; j += blockDim.x) {
    float num = 0.0f;
    for (int c = 0; c < nv; ++c)
      if (ml[2 * c] != -INFINITY) num += fast_exp2(ml[2 * c] - M) * po[(long long)c * D + j];
    a.out[head * D + j] = den > 0.0f ? num / den : 0.0f;
  }
}

}  // namespace

cudaError_t launch_combine(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  dim3 grid(a.num_q_heads, a.batch);
  combine_kernel<<<grid, head_dim, 0, stream>>>(a, head_dim);
  count_launch();
  return cudaGetLastError();
}

}  // namespace kvq
