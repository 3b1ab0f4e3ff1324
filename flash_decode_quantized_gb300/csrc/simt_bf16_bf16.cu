// CUDA-core decode kernels for K=BF16, V=BF16 (instantiations of kvq_decode_simt.cuh).
#include "kvq_decode_simt.cuh"

namespace kvq {
cudaError_t simt_launch_bf16_bf16(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  return simt::launch_pair<KVQ_CODEC_BF16, KVQ_CODEC_BF16>(a, head_dim, stream);
}
}  // namespace kvq
