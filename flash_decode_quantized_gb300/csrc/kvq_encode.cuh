// Encode of one K or V row into the paged store, shared by the append kernels and the
// decode kernel's fused append.
//
// One warp encodes one row (one token of one KV head).  Lane l holds elements
// [l*EPL, (l+1)*EPL) of the row, EPL = head_dim / 32, so a 32-element block spans
// 32/EPL adjacent lanes and its amax is a shuffle reduction inside that lane group.
// The arithmetic follows the codec contract exactly and is compiled without fast-math:
//   d = fp16_rn(amax / c) with an IEEE fp32 quotient, q = clamp(round_half_away(x / d), -c, c)
//   for the fp32 quotient x / d (reached exactly without a division per element, see
//   round_quotient_mag), q = 0 when d == 0.
#pragma once

#include <climits>

#include "kvq_internal.cuh"

namespace kvq {

// round_half_away(fp32(x / d)) for a bf16 value x and a normal fp16 scale d, without an
// IEEE division.  t = |x| * rcp(d) (rcp within 1 ulp) is within 2^-14 of the quotient
// y = |x| / d (|y| < 256).
// For normal d, y is either exactly on a rounding boundary k + 1/2 or at least 2^-12 away
// from it: x has 8 significant bits and (k + 1/2) d at most 19, so a nonzero
// |x - (k + 1/2) d| is at least min(ulp(x), ulp((k + 1/2) d)) >= 2^-12 d.  The fp32
// quotient (within 2^-16 of y) therefore rounds like y, and so does t except within
// 2^-12 of a boundary, where the exact residual |x| - (k + 1/2) d (an FMA of a 19-bit
// product, exact in fp32) decides, ties going away from zero.  Subnormal scales lack that
// separation and take the division.  Returns the magnitude; the caller applies the sign
// and the clamp.
__device__ __forceinline__ float round_quotient_mag(float ax, float d, float rcp_d) {
  const float at = ax * rcp_d;
  float aq = floorf(at + 0.5f);
  const float gap = at - (aq - 0.5f);            // distance above the lower boundary
  if (gap < 0x1p-12f) {
    if (fmaf(-(aq - 0.5f), d, ax) < 0.0f) aq -= 1.0f;   // below it: round down
  } else if (gap > 1.0f - 0x1p-12f) {
    if (fmaf(-(aq + 0.5f), d, ax) >= 0.0f) aq += 1.0f;  // on or above the upper one: up
  }
  return aq;
}

// fp32(amax / c) correctly rounded, for c = 127 or 7 and amax a finite bf16 value: the
// product by the rounded reciprocal and one FMA correction (Markstein's division step),
// which an exhaustive check over every positive finite bf16 amax finds equal to the IEEE
// quotient for both constants (tests/test_encode_quotient.py); infinities and NaNs pass
// through the product.
template <int C>
__device__ __forceinline__ float scale_quotient(float amax) {
  constexpr float r = 1.0f / C;                       // rounded reciprocal
  const float q0 = __fmul_rn(amax, r);
  const float e = fmaf(-q0, (float)C, amax);          // exact residual
  const float q1 = fmaf(e, r, q0);
  return amax <= 3.402823466e38f ? q1 : q0;
}

// Lane `lane`'s EPL elements of one bf16 row, as floats (exact).
// One vector load per lane (rows are 16-byte aligned: the bindings check it).
template <int EPL>
__device__ __forceinline__ void load_row(const __nv_bfloat16* __restrict__ row, int lane, float* x) {
  const __nv_bfloat16* src = row + lane * EPL;
  uint32_t w[EPL / 2];
  if constexpr (EPL == 2) {
    w[0] = *reinterpret_cast<const uint32_t*>(src);
  } else if constexpr (EPL == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    w[0] = v.x; w[1] = v.y;
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  }
#pragma unroll
  for (int k = 0; k < EPL / 2; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);               // bf16 -> fp32 is a shift
    x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

// Encodes one row (lane `lane` holds elements [lane*EPL, (lane+1)*EPL) in x) into store
// `st` at row r of page `page`, KV head h.  One warp; every lane takes part.
template <int CODEC, int EPL>
__device__ __forceinline__ void store_row(const StoreView& st, int page, int r, int h, const float* x) {
  constexpr int LANES_PER_BLOCK = kBlock / EPL;
  const int lane = threadIdx.x & 31;
  uint8_t* slab = const_cast<uint8_t*>(st.buf) + ((long long)page * st.num_kv_heads + h) * st.slab_bytes;
  if constexpr (CODEC == KVQ_CODEC_BF16 || CODEC == KVQ_CODEC_F16) {
    uint32_t w[EPL / 2];
#pragma unroll
    for (int k = 0; k < EPL / 2; ++k) {
      if constexpr (CODEC == KVQ_CODEC_BF16) {   // exact: x came from bf16
        __nv_bfloat162 v = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&v);
      } else {
        __half2 v = __floats2half2_rn(x[2 * k], x[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&v);
      }
    }
    uint8_t* dst = slab + (long long)r * st.row_bytes + lane * EPL * 2;
    if constexpr (EPL == 2) *reinterpret_cast<uint32_t*>(dst) = w[0];
    else if constexpr (EPL == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
    else *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    constexpr float C = (CODEC == KVQ_CODEC_Q8_0) ? 127.0f : 7.0f;
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int off = 1; off < LANES_PER_BLOCK; off <<= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const __half dh = __float2half_rn(scale_quotient<CODEC == KVQ_CODEC_Q8_0 ? 127 : 7>(amax));
    const float d = __half2float(dh);
    int qv[EPL];
    // warp-uniform choice, so the division path costs nothing when no block needs it
    if (__all_sync(0xffffffffu, d >= 0x1p-14f || d == 0.0f)) {
      float rcp_d;   // within 1 ulp of 1/d: t = |x| rcp_d stays within 2^-14 of the quotient
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rcp_d) : "f"(d));
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float aq = d == 0.0f ? 0.0f : round_quotient_mag(fabsf(x[e]), d, rcp_d);
        qv[e] = (int)copysignf(fminf(aq, C), x[e]);
      }
    } else {   // a subnormal scale somewhere in the row: IEEE quotients
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float t = d == 0.0f ? 0.0f : roundf(__fdiv_rn(x[e], d));
        qv[e] = (int)fminf(fmaxf(t, -C), C);
      }
    }
    uint8_t* dst = slab + (long long)r * st.row_bytes;
    // the lane's codes as one store: EPL bytes (q8_0) or EPL nibbles (q4s)
    if constexpr (CODEC == KVQ_CODEC_Q8_0) {
      // low bytes of the codes (two's complement) gathered by byte permutes
      uint32_t w[(EPL + 3) / 4];
#pragma unroll
      for (int k = 0; k < (EPL + 3) / 4; ++k) {
        const int e = 4 * k;
        if constexpr (EPL == 2) {
          w[k] = __byte_perm((uint32_t)qv[0], (uint32_t)qv[1], 0x0040);
        } else {
          w[k] = __byte_perm(__byte_perm((uint32_t)qv[e], (uint32_t)qv[e + 1], 0x0040),
                             __byte_perm((uint32_t)qv[e + 2], (uint32_t)qv[e + 3], 0x0040), 0x5410);
        }
      }
      if constexpr (EPL == 2) *reinterpret_cast<uint16_t*>(dst + lane * 2) = (uint16_t)w[0];
      else if constexpr (EPL == 4) *reinterpret_cast<uint32_t*>(dst + lane * 4) = w[0];
      else *reinterpret_cast<uint2*>(dst + lane * 8) = make_uint2(w[0], w[1]);
    } else {
      // sum_e (q_e + 8) 16^e: each term lies in [1, 15], so no nibble carries
      int acc = 0;
#pragma unroll
      for (int e = EPL - 1; e >= 0; --e) acc = acc * 16 + qv[e];
      constexpr uint32_t kEights = EPL == 2 ? 0x88u : EPL == 4 ? 0x8888u : 0x88888888u;
      const uint32_t w = (uint32_t)acc + kEights;
      if constexpr (EPL == 2) dst[lane] = (uint8_t)w;
      else if constexpr (EPL == 4) *reinterpret_cast<uint16_t*>(dst + lane * 2) = (uint16_t)w;
      else *reinterpret_cast<uint32_t*>(dst + lane * 4) = w;
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
  if (base < 0 || pos >= (long long)max_pages * st.page_size || pos >= (long long)INT_MAX) {
    if (lane == 0) record_fault(st.status, KVQ_DEVICE_BAD_POSITION);
    return;
  }
  // positions fit in 32 bits here (the table holds fewer than 2^31 slots): 32-bit division
  const int page = page_table[(long long)b * max_pages + (int)pos / st.page_size];
  if (page < 0 || page >= st.num_pages) {
    if (lane == 0) record_fault(st.status, KVQ_DEVICE_BAD_PAGE);
    return;
  }
  float x[EPL];
  load_row<EPL>(rows + row_id * D, lane, x);
  store_row<CODEC, EPL>(st, page, (int)pos % st.page_size, h, x);
}

}  // namespace kvq
