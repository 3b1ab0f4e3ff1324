// Device helpers shared by the decode kernels: cp.async staging, exp2, row dequant.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

__device__ __forceinline__ float fast_exp2(float x) {
  // ex2.approx: hardware base-2 exponential, |rel err| ~ 2^-22; ex2(-inf) = +0.
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// Converts 16 consecutive stored elements of a row (starting at `p`, 16-byte aligned in
// shared memory for 8-bit and 16-bit rows, 8-byte aligned for 4-bit rows) to floats.
// Quantized codecs yield the integer codes; the caller applies the block scale.
template <int CODEC>
__device__ __forceinline__ void load16(const uint8_t* p, float* out) {
  if constexpr (CODEC == KVQ_CODEC_Q8_0) {
    const int4 w = *reinterpret_cast<const int4*>(p);
    const int ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) out[4 * i + k] = (float)(int8_t)((ws[i] >> (8 * k)) & 0xff);
  } else if constexpr (CODEC == KVQ_CODEC_Q4S) {
    const int2 w = *reinterpret_cast<const int2*>(p);
    const int ws[2] = {w.x, w.y};
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int k = 0; k < 8; ++k) out[8 * i + k] = (float)(((ws[i] >> (4 * k)) & 0xf) - 8);
  } else {
    const int4 w0 = *reinterpret_cast<const int4*>(p);
    const int4 w1 = *reinterpret_cast<const int4*>(p + 16);
    const uint32_t ws[8] = {(uint32_t)w0.x, (uint32_t)w0.y, (uint32_t)w0.z, (uint32_t)w0.w,
                            (uint32_t)w1.x, (uint32_t)w1.y, (uint32_t)w1.z, (uint32_t)w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if constexpr (CODEC == KVQ_CODEC_BF16) {
        out[2 * i] = __uint_as_float(ws[i] << 16);
        out[2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
      } else {
        const __half2 h = *reinterpret_cast<const __half2*>(&ws[i]);
        const float2 f = __half22float2(h);
        out[2 * i] = f.x;
        out[2 * i + 1] = f.y;
      }
    }
  }
}

// Converts N (2, 4 or 8) consecutive stored elements starting at element `e0` of a row.
template <int CODEC, int N>
__device__ __forceinline__ void load_n(const uint8_t* row, int e0, float* out) {
  if constexpr (CODEC == KVQ_CODEC_Q8_0) {
#pragma unroll
    for (int k = 0; k < N; ++k) out[k] = (float)(int8_t)row[e0 + k];
  } else if constexpr (CODEC == KVQ_CODEC_Q4S) {
#pragma unroll
    for (int k = 0; k < N; k += 2) {
      const int byte = row[(e0 + k) >> 1];
      out[k] = (float)((byte & 0xf) - 8);
      out[k + 1] = (float)((byte >> 4) - 8);
    }
  } else if constexpr (CODEC == KVQ_CODEC_BF16) {
    const uint16_t* r = reinterpret_cast<const uint16_t*>(row);
#pragma unroll
    for (int k = 0; k < N; ++k) out[k] = __uint_as_float(((uint32_t)r[e0 + k]) << 16);
  } else {
    const __half* r = reinterpret_cast<const __half*>(row);
#pragma unroll
    for (int k = 0; k < N; ++k) out[k] = __half2float(r[e0 + k]);
  }
}

constexpr bool is_quant(int codec) { return codec == KVQ_CODEC_Q8_0 || codec == KVQ_CODEC_Q4S; }

}  // namespace kvq
