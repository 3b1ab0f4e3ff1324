// CUDA-core decode kernels for K=F16, V=F16 (instantiations of kvq_decode_simt.cuh).
#include "kvq_decode_simt.cuh"

namespace kvq {
cudaError_t simt_launch_f16_f16(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  return simt::launch_pair<KVQ_CODEC_F16, KVQ_CODEC_F16>(a, head_dim, stream);
}
}  // namespace kvq
