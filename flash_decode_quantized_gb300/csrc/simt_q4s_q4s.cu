// CUDA-core decode kernels for K=Q4S, V=Q4S (instantiations of kvq_decode_simt.cuh).
#include "kvq_decode_simt.cuh"

namespace kvq {
cudaError_t simt_launch_q4s_q4s(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  return simt::launch_pair<KVQ_CODEC_Q4S, KVQ_CODEC_Q4S>(a, head_dim, stream);
}
}  // namespace kvq
