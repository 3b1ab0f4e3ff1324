// CUDA-core decode kernels for K=Q4S, V=BF16 (instantiations of kvq_decode_simt.cuh).
#include "kvq_decode_simt.cuh"

namespace kvq {
cudaError_t simt_launch_q4s_bf16(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  return simt::launch_pair<KVQ_CODEC_Q4S, KVQ_CODEC_BF16>(a, head_dim, stream);
}
}  // namespace kvq
