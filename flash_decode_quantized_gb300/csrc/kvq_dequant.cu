// Separate dequantize pass: a quantized store's rows rewritten as a 16-bit store.
//
// This is the comparison arm, not the hot path: halobench record clm-0022 (METHOD, depth
// tables) attributes the quantized-KV decode penalty of the stock build to converting
// the quantized cache outside the attention kernel instead of on load; the penalty grows
// with depth.  kvq_dequantize + a 16-bit kvq_flash_decode reproduces that arm so the
// fused kernel can be measured against it on the same data.
//
// One CTA per (page slot j of sequence b, KV head): rows [0, n) of the slab, n the part of
// seq_lens[b] that falls in page j.  A thread writes 16 bytes (8 elements) at a time:
// x = d * q exactly in fp32 (11-bit scale times a code of at most 8 bits), rounded once to
// the 16-bit type.

#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int kDequantThreads = 256;

template <bool F16>
__device__ __forceinline__ uint32_t pack16x2(float a, float b) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <int SRC, bool F16>
__global__ void __launch_bounds__(kDequantThreads)
dequant_kernel(StoreView src, StoreView dst, const int32_t* __restrict__ seq_lens,
               const int32_t* __restrict__ page_table, int max_pages, int head_dim) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int j = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int P = src.page_size;
  const long long L = seq_lens[b];
  const long long n_ll = L - (long long)j * P;
  if (n_ll <= 0) return;
  if (L > (long long)max_pages * P) {   // rows past the table: recorded, nothing written
    if (threadIdx.x == 0 && j == 0 && h == 0) record_fault(dst.status, KVQ_DEVICE_BAD_SEQ_LEN);
    return;
  }
  const int n = n_ll < P ? (int)n_ll : P;
  const int page = page_table[(long long)b * max_pages + j];
  if (page < 0 || page >= src.num_pages || page >= dst.num_pages) {
    if (threadIdx.x == 0) record_fault(dst.status, KVQ_DEVICE_BAD_PAGE);
    return;
  }
  const uint8_t* s_slab = src.buf + ((long long)page * src.num_kv_heads + h) * src.slab_bytes;
  uint8_t* d_slab = const_cast<uint8_t*>(dst.buf) + ((long long)page * dst.num_kv_heads + h) * dst.slab_bytes;
  const __half* s_scales = reinterpret_cast<const __half*>(s_slab + (long long)P * src.row_bytes);
  const int groups = head_dim / 8;   // 16-byte output groups per row
  for (int idx = threadIdx.x; idx < n * groups; idx += kDequantThreads) {
    const int r = idx / groups, g = idx % groups;
    const int e0 = 8 * g;
    const float d = __half2float(s_scales[(long long)r * src.n_scales + e0 / kBlock]);
    float x[8];
    if constexpr (SRC == KVQ_CODEC_Q8_0) {
      const uint2 w = *reinterpret_cast<const uint2*>(s_slab + (long long)r * src.row_bytes + e0);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[e] = d * (float)(int8_t)(w.x >> (8 * e));
        x[4 + e] = d * (float)(int8_t)(w.y >> (8 * e));
      }
    } else {   // q4s: 8 nibbles, element 2k low nibble of byte k
      const uint32_t w = *reinterpret_cast<const uint32_t*>(s_slab + (long long)r * src.row_bytes + e0 / 2);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = d * (float)((int)((w >> (4 * e)) & 15u) - 8);
    }
    uint4 o;
    o.x = pack16x2<F16>(x[0], x[1]);
    o.y = pack16x2<F16>(x[2], x[3]);
    o.z = pack16x2<F16>(x[4], x[5]);
    o.w = pack16x2<F16>(x[6], x[7]);
    *reinterpret_cast<uint4*>(d_slab + (long long)r * dst.row_bytes + 2 * e0) = o;
  }
}

template <int SRC>
cudaError_t launch_src(const kvq_store* src, kvq_store* dst, const int32_t* seq_lens,
                       const int32_t* page_table, int max_pages, int batch, cudaStream_t stream) {
  const dim3 grid(max_pages, src->desc.num_kv_heads, batch);
  const StoreView s = view_of(src), d = view_of(dst);
  cudaError_t e;
  if (dst->desc.codec == KVQ_CODEC_F16)
    e = launch_pdl(dequant_kernel<SRC, true>, grid, dim3(kDequantThreads), 0, stream, s, d, seq_lens, page_table,
                   max_pages, src->desc.head_dim);
  else
    e = launch_pdl(dequant_kernel<SRC, false>, grid, dim3(kDequantThreads), 0, stream, s, d, seq_lens, page_table,
                   max_pages, src->desc.head_dim);
  count_launch();
  return e;
}

}  // namespace

cudaError_t launch_dequantize(const kvq_store* src, kvq_store* dst, const int32_t* seq_lens,
                              const int32_t* page_table, int max_pages, int batch, cudaStream_t stream) {
  return src->desc.codec == KVQ_CODEC_Q8_0
             ? launch_src<KVQ_CODEC_Q8_0>(src, dst, seq_lens, page_table, max_pages, batch, stream)
             : launch_src<KVQ_CODEC_Q4S>(src, dst, seq_lens, page_table, max_pages, batch, stream);
}

}  // namespace kvq
