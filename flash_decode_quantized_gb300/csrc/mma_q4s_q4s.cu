// Tensor-core decode kernels for K=Q4S, V=Q4S (instantiations of kvq_decode_mma.cuh).
#include "kvq_decode_mma.cuh"

namespace kvq {
cudaError_t mma_launch_q4s_q4s(const DecodeArgs& a, int head_dim, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, cudaStream_t stream) {
  return mma::launch_pair<KVQ_CODEC_Q4S, KVQ_CODEC_Q4S>(a, head_dim, tmk, tmv, stream);
}
int mma_occupancy_q4s_q4s(int head_dim, int group, int* pipes, int solo) {
  return mma::occupancy_pair<KVQ_CODEC_Q4S, KVQ_CODEC_Q4S>(head_dim, group, pipes, solo != 0);
}
}  // namespace kvq
