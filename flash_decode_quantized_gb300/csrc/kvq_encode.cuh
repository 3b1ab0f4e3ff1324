// Encode of one K or V row into the paged store, shared by the append kernels and the
// decode kernel's fused append.
//
// One warp encodes one row (one token of one KV head).  Lane l holds elements
// [l*EPL, (l+1)*EPL) of the row, EPL = head_dim / 32, so a 32-element block spans
// 32/EPL adjacent lanes and its amax is a shuffle reduction inside that lane group.
// The arithmetic follows the codec contract exactly and is compiled without fast-math:
//   d = fp16_rn(amax / c) with an IEEE fp32 quotient, q = clamp(roundf(x / d), -c, c)
//   (roundf rounds half away from zero), q = 0 when d == 0.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

// Lane `lane`'s EPL elements of one bf16 row, as floats (exact).
template <int EPL>
__device__ __forceinline__ void load_row(const __nv_bfloat16* __restrict__ row, int lane, float* x) {
  const __nv_bfloat16* src = row + lane * EPL;
#pragma unroll
  for (int e = 0; e < EPL; ++e) x[e] = __bfloat162float(src[e]);
}

// Encodes one row (lane `lane` holds elements [lane*EPL, (lane+1)*EPL) in x) into store
// `st` at row r of page `page`, KV head h.  One warp; every lane takes part.
template <int CODEC, int EPL>
__device__ __forceinline__ void store_row(const StoreView& st, int page, int r, int h, const float* x) {
  constexpr int LANES_PER_BLOCK = kBlock / EPL;
  const int lane = threadIdx.x & 31;
  uint8_t* slab = const_cast<uint8_t*>(st.buf) + ((long long)page * st.num_kv_heads + h) * st.slab_bytes;
  if constexpr (CODEC == KVQ_CODEC_BF16) {
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(slab + (long long)r * st.row_bytes) + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[e] = __float2bfloat16_rn(x[e]);   // exact: x came from bf16
  } else if constexpr (CODEC == KVQ_CODEC_F16) {
    __half* dst = reinterpret_cast<__half*>(slab + (long long)r * st.row_bytes) + lane * EPL;
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[e] = __float2half_rn(x[e]);
  } else {
    constexpr float C = (CODEC == KVQ_CODEC_Q8_0) ? 127.0f : 7.0f;
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int off = 1; off < LANES_PER_BLOCK; off <<= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const __half dh = __float2half_rn(__fdiv_rn(amax, C));
    const float d = __half2float(dh);
    int qv[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      float t = (d == 0.0f) ? 0.0f : roundf(__fdiv_rn(x[e], d));
      t = fminf(fmaxf(t, -C), C);
      qv[e] = (int)t;
    }
    uint8_t* dst = slab + (long long)r * st.row_bytes;
    if constexpr (CODEC == KVQ_CODEC_Q8_0) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) dst[lane * EPL + e] = (uint8_t)(int8_t)qv[e];
    } else {
#pragma unroll
      for (int e = 0; e < EPL; e += 2)
        dst[(lane * EPL + e) / 2] = (uint8_t)((qv[e] + 8) | ((qv[e + 1] + 8) << 4));
    }
    if ((lane % LANES_PER_BLOCK) == 0) {
      __half* sc = reinterpret_cast<__half*>(slab + (long long)st.page_size * st.row_bytes) +
                   (long long)r * st.n_scales + (lane * EPL) / kBlock;
      *sc = dh;
    }
  }
}

// Encodes row `row_id` of `rows` ([batch][n_new][Hkv][D]) into store `st` at position
// base + i, where (b, i, h) are the row's coordinates and base = seq_lens[b].  One warp.
// An invalid position or page is recorded as a device fault and the row is skipped.
template <int CODEC, int EPL>
__device__ __forceinline__ void encode_row(const StoreView& st, const __nv_bfloat16* __restrict__ rows,
                                           long long row_id, int n_new, long long base, int b, int i, int h,
                                           const int32_t* __restrict__ page_table, int max_pages) {
  constexpr int D = EPL * 32;
  const int lane = threadIdx.x & 31;
  const long long pos = base + i;
  if (base < 0 || pos >= (long long)max_pages * st.page_size) {
    if (lane == 0) record_fault(st.status, KVQ_DEVICE_BAD_POSITION);
    return;
  }
  const int page = page_table[(long long)b * max_pages + pos / st.page_size];
  if (page < 0 || page >= st.num_pages) {
    if (lane == 0) record_fault(st.status, KVQ_DEVICE_BAD_PAGE);
    return;
  }
  float x[EPL];
  load_row<EPL>(rows + row_id * D, lane, x);
  store_row<CODEC, EPL>(st, page, (int)(pos % st.page_size), h, x);
}

}  // namespace kvq
