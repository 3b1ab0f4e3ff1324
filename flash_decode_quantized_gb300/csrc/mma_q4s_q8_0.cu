// Tensor-core decode kernels for K=Q4S, V=Q8_0 (instantiations of kvq_decode_mma.cuh).
#include "kvq_decode_mma.cuh"

namespace kvq {
cudaError_t mma_launch_q4s_q8_0(const DecodeArgs& a, int head_dim, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, cudaStream_t stream) {
  return mma::launch_pair<KVQ_CODEC_Q4S, KVQ_CODEC_Q8_0>(a, head_dim, tmk, tmv, stream);
}
int mma_occupancy_q4s_q8_0(int head_dim, int group, int* pipes, int solo) {
  return mma::occupancy_pair<KVQ_CODEC_Q4S, KVQ_CODEC_Q8_0>(head_dim, group, pipes, solo != 0);
}
}  // namespace kvq
