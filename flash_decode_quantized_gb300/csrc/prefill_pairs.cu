// Prefill attention kernels for the K/V codec pairs that have them: the tensor-core
// (tcgen05) kernel of kvq_prefill_tc.cuh for the eight decode pairs plus q8_0/f16 and
// f16/q8_0 at head_dim 128, the warp-MMA kernel of kvq_prefill.cuh at head_dim 64 and 256.
#include "kvq_prefill.cuh"
#include "kvq_prefill_tc.cuh"

namespace kvq {
cudaError_t prefill_launch(int kc, int vc, const PrefillArgs& a, int batch, int head_dim,
                           const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream) {
  using namespace prefill;
  if (head_dim == 128) {
    constexpr int Q8 = KVQ_CODEC_Q8_0, F16 = KVQ_CODEC_F16;
    if (kc == Q8 && vc == Q8) return prefill_tc::launch<Q8, Q8>(a, batch, tmk, tmv, stream);
    if (kc == F16 && vc == F16) return prefill_tc::launch<F16, F16>(a, batch, tmk, tmv, stream);
    if (kc == Q8 && vc == F16) return prefill_tc::launch<Q8, F16>(a, batch, tmk, tmv, stream);
    if (kc == F16 && vc == Q8) return prefill_tc::launch<F16, Q8>(a, batch, tmk, tmv, stream);
    constexpr int BF = KVQ_CODEC_BF16;
    if (kc == BF && vc == BF) return prefill_tc::launch<BF, BF>(a, batch, tmk, tmv, stream);
    if (kc == Q8 && vc == BF) return prefill_tc::launch<Q8, BF>(a, batch, tmk, tmv, stream);
    constexpr int Q4 = KVQ_CODEC_Q4S;
    if (kc == Q4 && vc == Q4) return prefill_tc::launch<Q4, Q4>(a, batch, tmk, tmv, stream);
    if (kc == Q8 && vc == Q4) return prefill_tc::launch<Q8, Q4>(a, batch, tmk, tmv, stream);
    if (kc == Q4 && vc == Q8) return prefill_tc::launch<Q4, Q8>(a, batch, tmk, tmv, stream);
    if (kc == Q4 && vc == BF) return prefill_tc::launch<Q4, BF>(a, batch, tmk, tmv, stream);
  }
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
