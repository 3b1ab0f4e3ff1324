// Tensor-core decode kernels for K=BF16, V=BF16 (instantiations of kvq_decode_mma.cuh).
#include "kvq_decode_mma.cuh"

namespace kvq {
cudaError_t mma_launch_bf16_bf16(const DecodeArgs& a, int head_dim, const CUtensorMap& tmk,
                            const CUtensorMap& tmv, cudaStream_t stream) {
  return mma::launch_pair<KVQ_CODEC_BF16, KVQ_CODEC_BF16>(a, head_dim, tmk, tmv, stream);
}
int mma_occupancy_bf16_bf16(int head_dim, int group, int* pipes, int solo) {
  return mma::occupancy_pair<KVQ_CODEC_BF16, KVQ_CODEC_BF16>(head_dim, group, pipes, solo != 0);
}
}  // namespace kvq
