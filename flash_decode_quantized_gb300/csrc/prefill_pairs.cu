// Prefill attention kernels for the K/V codec pairs that have them (instantiations of
// kvq_prefill.cuh).
#include "kvq_prefill.cuh"

namespace kvq {
cudaError_t prefill_launch(int kc, int vc, const PrefillArgs& a, int batch, int head_dim,
                           const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream) {
  using namespace prefill;
  if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_Q8_0) return launch_pair<KVQ_CODEC_Q8_0, KVQ_CODEC_Q8_0>(a, batch, head_dim, tmk, tmv, stream);
  if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_Q4S) return launch_pair<KVQ_CODEC_Q4S, KVQ_CODEC_Q4S>(a, batch, head_dim, tmk, tmv, stream);
  if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_Q4S) return launch_pair<KVQ_CODEC_Q8_0, KVQ_CODEC_Q4S>(a, batch, head_dim, tmk, tmv, stream);
  if (kc == KVQ_CODEC_F16 && vc == KVQ_CODEC_F16) return launch_pair<KVQ_CODEC_F16, KVQ_CODEC_F16>(a, batch, head_dim, tmk, tmv, stream);
  if (kc == KVQ_CODEC_BF16 && vc == KVQ_CODEC_BF16) return launch_pair<KVQ_CODEC_BF16, KVQ_CODEC_BF16>(a, batch, head_dim, tmk, tmv, stream);
  if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_BF16) return launch_pair<KVQ_CODEC_Q8_0, KVQ_CODEC_BF16>(a, batch, head_dim, tmk, tmv, stream);
  if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_Q8_0) return launch_pair<KVQ_CODEC_Q4S, KVQ_CODEC_Q8_0>(a, batch, head_dim, tmk, tmv, stream);
  if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_BF16) return launch_pair<KVQ_CODEC_Q4S, KVQ_CODEC_BF16>(a, batch, head_dim, tmk, tmv, stream);
  return cudaErrorNotSupported;
}
}  // namespace kvq
