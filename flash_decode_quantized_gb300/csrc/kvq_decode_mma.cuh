// Tensor-core split-K flash-decode with dequantization fused into the QK^T and PV loops.
//
// Same computation and split as the CUDA-core kernel (the "flash-decode-over-quant"
// class of rMLX issue #292, with halobench record clm-0022's "dequantize KV on load"):
// quantized K/V tiles are staged in shared memory exactly as stored and converted in
// registers right before the matrix instructions that consume them.
//
// Why tensor cores: the CUDA-core kernel issues ~3.3k lane-instructions per (token, KV
// head) for q8_0 at GQA 4:1, which caps it near half of HBM bandwidth even at full issue
// rate.  Here the two contractions run on mma.sync m16n8k16 (fp32 accumulate):
//
//  * QK^T, tokens on M: S[t, h] = sum_b d_k[t, b] * sum_{j in b} k_int[t, j] * q[h, j].
//    A = the stored K rows of 16 tokens, read with ldmatrix and turned into exact f16
//    integers in registers; B = q (N = 8 heads of the group).  Each 32-element block's
//    two k16 steps accumulate into a fresh fragment that is then scaled by d_k (and
//    the softmax scale) and added to S, so the block scale is applied once per block.
//    The k order inside a 16-element step is permuted to match the bytes ldmatrix
//    hands each lane; q is laid out with the same permutation.
//  * PV, head_dim on M: O^T[j, c] += sum_t v_int[t, j] * P[t, c].  A = the stored V rows
//    (ldmatrix.trans, converted the same way), B = the probabilities.  The V block scale
//    d_v[t, b] varies along the contraction, so it is folded into B per block:
//    P_b[t, h] = p[t, h] * d_v[t, b] * 2^(kPScale - E).  To keep fp32-level accuracy from
//    16-bit operands P_b is split into hi + lo halves (hi = f16(x), lo = f16(x - hi));
//    with at most 4 heads per warp the hi and lo parts occupy the 8 N columns of one
//    MMA, so the split costs no extra tensor instructions.  E is a running power-of-two
//    bound of the V scales seen so far (like the running max of the softmax), which
//    keeps P_b inside the f16 range whatever the magnitude of V.
//
// Data movement: one elected thread streams 64-token tiles of one (page, head) slab with
// TMA (cp.async.bulk.tensor, 128/64/32-byte swizzle so the ldmatrix reads are free of
// bank conflicts) plus bulk copies of the fp16 scales into an NS-deep ring of stages
// guarded by mbarriers (full: copies landed; empty: every warp is done with the stage);
// the warps take 16 tokens of every tile each and keep their
// own online-softmax state (running max m and sum l per head, base 2).  Every wait is
// bounded: on timeout the kernel records KVQ_DEVICE_TIMEOUT and returns.
//
// GQA: one CTA serves all heads of a KV head's group from each tile; groups of more than
// 8 heads are split over warp groups (8 heads each) that read the same tiles.
#pragma once

#include <cuda.h>

#include "kvq_device.cuh"
#include "kvq_encode.cuh"

namespace kvq {
namespace mma {

constexpr int kT = 64;            // tokens per stage
constexpr int kTimeoutIters = 1 << 22;
// Lazy online softmax: scores are exponentiated against a warp-uniform reference max
// that is raised only when a score exceeds it by more than kLazy (log2 units), so every
// p stays <= 2^kLazy and most tiles need no cross-lane reduction.
constexpr float kLazy = 8.0f;
// P_b = p * d_v * 2^(kPScale - E) <= 2^(kLazy + kPScale) = 2^14 fits f16 (max 65504).
constexpr int kPScale = 6;

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Release of a stage by one of `warps` warps: lane 0 arrives on the stage's empty barrier
// and counts the release; true (in every lane) for the warp whose release is the last
// one, which also returns the count to zero.
__device__ __forceinline__ bool release_last(uint32_t bar_empty, unsigned* cnt, int lane, int warps) {
  uint32_t old = 0u;
  asm volatile("{\n .reg .pred p;\n setp.eq.s32 p, %2, 0;\n"
               " @p mbarrier.arrive.shared::cta.b64 _, [%1];\n"
               " @p atom.shared::cta.add.u32 %0, [%3], 1;\n}\n"
               : "+r"(old) : "r"(bar_empty), "r"(lane), "r"((uint32_t)__cvta_generic_to_shared(cnt)) : "memory");
  const bool last = __shfl_sync(0xffffffffu, old, 0) == (uint32_t)(warps - 1);
  if (last && lane == 0) atomicExch(cnt, 0u);
  return last;
}
__device__ __forceinline__ uint32_t mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(done) : "r"(bar), "r"(parity) : "memory");
  return done;
}
// Bounded wait, by every lane of a warp, for the phase of parity `parity` to complete.
// Each lane observes the completion itself (acquire); the result is warp-uniform, so
// the warp leaves together.  False on timeout.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, int limit = kTimeoutIters) {
  for (int it = 0; it < limit; ++it)
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
  return false;
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            int c3, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// L2 policy for data a call reads exactly once (the KV stream): evict first, so that the
// stream does not push out of L2 what is reused (the kernel's code, the split partials,
// the page table and lengths).
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_4d_ef(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                               int c3, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_load_ef(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                             uint64_t policy) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}
__device__ __forceinline__ uint32_t movtrans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
template <bool BF16>
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if constexpr (BF16) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// ---------------------------------------------------------------- conversions

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t x, uint32_t y) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<__half2*>(&y));
  return *reinterpret_cast<uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t x, uint32_t y, uint32_t z) {
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), *reinterpret_cast<__half2*>(&y),
                      *reinterpret_cast<__half2*>(&z));
  return *reinterpret_cast<uint32_t*>(&r);
}
// Magic-number conversion of integer codes to f16: the bits 0x64 << 8 | u encode the
// f16 value 1024 + u exactly (u < 1024).  V operands subtract the constant offset in f16
// registers (exact); K operands keep it and the QK accumulator is seeded with
// -offset * sum(q) of the block (kBias8 / kBias4K), so the offset must stay small
// against the dot product it rides on.
//
// Signed bytes packed in `u_biased` (each byte already XORed with 0x80, i.e. q + 128)
// to the f16 pair (1152 + q) of the two bytes named by `sel` (0x4X4Y picks bytes X, Y).
__device__ __forceinline__ uint32_t i8pair_raw(uint32_t u_biased, uint32_t sel) {
  return __byte_perm(u_biased, 0x64646464u, sel);
}
// (a & b) | c as one lop3 (truth table 0xEA) with b and c in registers: written as C the
// mask-and-insert compiled to two instructions (4-bit K+V decode 41.5 -> 38.1 us at the
// 65536-token headline shape).
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
// Nibble pair (bits 0-3 and 16-19 of w) holding u = q + 8 -> the f16 pair (1032 + q).
__device__ __forceinline__ uint32_t u4pair_raw(uint32_t w) {
  return and_or(w, 0x000F000Fu, 0x64006400u);
}
// Nibble pair (bits 4-7 and 20-23 of w) holding u = q + 8 -> the f16 pair (1024 + 16 u), with
// no shift: hfma2_u32(x, 1/16, -72) then gives q exactly (64 + u - 72, one rounding of an
// exact small integer).
__device__ __forceinline__ uint32_t u4pair_hi_raw(uint32_t w) {
  return and_or(w, 0x00F000F0u, 0x64006400u);
}
constexpr uint32_t kSixteenth2 = 0x2C002C00u;   // f16 pair (1/16, 1/16)
constexpr uint32_t kMinus72x2 = 0xD480D480u;    // f16 pair (-72, -72)
// Nibble pair (bits 4-7 and 20-23 of w) holding u = q + 8 -> the f16 pair 8 + u/8 =
// 9 + q/8 (0x48 << 8 is 8.0; the nibble lands in mantissa bits 4-7, so a word's nibbles
// need shifts by 4, 0, -4 and -8 bits: three shifts and four lop3s per word).  The K
// codes of the 4-bit codec use this form: its offset is ~10x a code's step, as for the
// 8-bit codes; with the 1024-based one (offset ~150x the step) the seeded accumulator
// carried ~1000x the block's dot product and the tensor-core accumulate lost its low bits
// (score errors ~1e-3 in log2 units for keys of magnitude ~50).
__device__ __forceinline__ uint32_t u4pair_half(uint32_t w) {
  return and_or(w, 0x00F000F0u, 0x48004800u);
}
constexpr float kBias8 = 1152.0f;            // offset of i8pair_raw values
constexpr float kBias4K = 9.0f;              // offset of u4pair_half values (which carry q/8)
constexpr float kScale4K = 8.0f;             // u4pair_half values carry q/8

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  if constexpr (BF16) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v));
  } else {
    return __half22float2(*reinterpret_cast<__half2*>(&v));
  }
}
// y = x + k * h for the two 16-bit halves h of hp (k a 16-bit constant): one mixed-precision
// FMA per value, exact for k = -1 when h is x rounded (Sterbenz).
template <bool BF16>
__device__ __forceinline__ void add_k_times(uint32_t hp, unsigned short k, float x0, float x1, float& y0, float& y1) {
  if constexpr (BF16)
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n fma.rn.f32.bf16 %0, l, %3, %4;\n fma.rn.f32.bf16 %1, h, %3, %5;\n}"
        : "=f"(y0), "=f"(y1) : "r"(hp), "h"(k), "f"(x0), "f"(x1));
  else
    asm("{\n .reg .b16 l, h;\n mov.b32 {l, h}, %2;\n fma.rn.f32.f16 %0, l, %3, %4;\n fma.rn.f32.f16 %1, h, %3, %5;\n}"
        : "=f"(y0), "=f"(y1) : "r"(hp), "h"(k), "f"(x0), "f"(x1));
}
// x -> (hi, lo) pairs with hi = round(x), lo = round(x - hi), for two values.
template <bool BF16>
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  hi = pack2<BF16>(x0, x1);
  float y0, y1;
  add_k_times<BF16>(hi, BF16 ? 0xBF80 : 0xBC00, x0, x1, y0, y1);
  lo = pack2<BF16>(y0, y1);
}

// (x0, x1) -> f16/bf16 pair of x (neg_sel = 0: the hi part) or of x - hi (neg_sel = -1).
template <bool BF16>
__device__ __forceinline__ uint32_t hi_or_lo(float x0, float x1, unsigned short neg_sel) {
  float y0, y1;
  add_k_times<BF16>(pack2<BF16>(x0, x1), neg_sel, x0, x1, y0, y1);
  return pack2<BF16>(y0, y1);
}

// The NB fp16 scales of tile row t (a contiguous NB*2-byte run) as NB/2 packed words.
template <int NB>
__device__ __forceinline__ void load_scale_words(const uint8_t* base, int t, uint32_t* w) {
  const uint8_t* p = base + t * NB * 2;
  if constexpr (NB == 2) {
    w[0] = *reinterpret_cast<const uint32_t*>(p);
  } else if constexpr (NB == 4) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    w[0] = v.x; w[1] = v.y;
  } else {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
  }
}

// ---------------------------------------------------------------- layout

// SOLO: one 4-warp pipeline per CTA and up to four CTAs per SM, for grids of many short
// CTAs (more (sequence, KV head) units than SMs), whose prologues and merges then overlap.
template <int KC, int VC, int D, int GW, int HG, bool SOLO = false>
struct Cfg {
  // Heads on M (GW == 16, kvq_decode_hm.cuh): warps of 16 query rows x 16 tokens, HG row
  // groups per pipeline.
  static constexpr bool HM = GW == 16;
  static constexpr int PW = 4 * HG;                       // warps per pipeline (4 per head group)
  static constexpr int NPV = GW <= 4 ? 1 : 2;             // PV n-tiles per warp
  static constexpr bool KBF = KC == KVQ_CODEC_BF16;       // MMA type of QK^T
  static constexpr bool VBF = VC == KVQ_CODEC_BF16;       // MMA type of PV
  static constexpr bool KQ = is_quant(KC), VQ = is_quant(VC);
  static constexpr int KRB = KC == KVQ_CODEC_Q8_0 ? D : KC == KVQ_CODEC_Q4S ? D / 2 : 2 * D;
  static constexpr int VRB = VC == KVQ_CODEC_Q8_0 ? D : VC == KVQ_CODEC_Q4S ? D / 2 : 2 * D;
  static constexpr int NB = D / kBlock;                   // blocks per row
  static constexpr int KLINE = KRB >= 128 ? 128 : KRB;    // TMA box width / swizzle span
  static constexpr int VLINE = VRB >= 128 ? 128 : VRB;
  static constexpr int al1k(int x) { return (x + 1023) / 1024 * 1024; }
  // stage: [K rows | V rows | K scales | V scales]; row regions 1024-aligned (swizzle)
  static constexpr int KROWS = al1k(kT * KRB);
  static constexpr int VROWS = al1k(kT * VRB);
  static constexpr int KSC = KQ ? kT * NB * 2 : 0;        // multiples of 16 bytes
  static constexpr int VSC = VQ ? kT * NB * 2 : 0;
  static constexpr int V_OFF = KROWS, KSC_OFF = KROWS + VROWS, VSC_OFF = KSC_OFF + KSC;
  static constexpr int STAGE = al1k(KROWS + VROWS + KSC + VSC);
  // Four pipelines per CTA (one CTA per SM, 16 warps) for 4-head warps when two stages
  // fit a quarter of the SM's shared memory: registers capped at 128 (no spills at
  // D <= 128).  Each pipeline is 4 warps with its own ring of stages; the CTA merges its
  // pipelines in shared memory, so a split has a quarter as many partials as with one
  // pipeline per CTA.  Otherwise one pipeline per CTA and register use sets occupancy.
  static constexpr bool PACK = !SOLO && HG == 1 && GW <= 4 && D <= 128 && 2 * STAGE + 6 * 1024 <= 56 * 1024;
  // HM: for one row group two pipelines per CTA at head_dim 256 (8 warps per SM at up to
  // 255 registers: the O accumulators alone take D / 2) and three at head_dim 128 (12
  // warps at 168 registers, no spills: 54 -> 47 us for GQA 16:1 at 65536 tokens, 8 KV
  // heads); one pipeline for two row groups.  8-head warps at head_dim <= 128: three
  // pipelines (12 warps at 168 registers instead of two CTAs of 4 warps at 223: GQA 8:1 at
  // 65536 tokens 48 -> 43.6 us for q8_0, 50 -> 45 us for q4s; four pipelines gain nothing).
  // 4-head warps at head_dim 256 where two stages of each of three pipelines fit: three
  // (8192 tokens 24.9 -> 20.6 us, one KV head at 131072 tokens 34.8 -> 31.6 us)
  static constexpr int NP = PACK ? 4 : (HM && HG == 1) ? (D == 128 ? 3 : 2)
                          : ((GW == 8 && D <= 128) || (GW == 4 && D == 256 && !SOLO && 6 * STAGE <= 210 * 1024)) && HG == 1
                              ? 3 : 1;   // pipelines per CTA
  // the lean tile loop (see decode_cta) serves warps of at most 4 heads at D <= 128
  static constexpr bool LEAN = HG == 1 && GW <= 4 && D <= 128;
  static constexpr int NW = PW * NP;                      // warps per CTA
  static constexpr int THREADS = NW * 32;
  static constexpr int MINB = SOLO ? 4 : 1;
  // ring depth per pipeline: as many stages (2..4) as fit the per-pipeline budget
  static constexpr int SMEM_BUDGET = HM ? (HG > 1 ? 204 * 1024 : 104 * 1024 + 2048)
                                     : HG > 1 ? 200 * 1024 : D == 256 ? 100 * 1024 : (PACK || SOLO) ? 54 * 1024 : 70 * 1024;
  static constexpr int NS0 = (SMEM_BUDGET - 2048) / STAGE;
  static constexpr int NS = NS0 > 4 ? 4 : (NS0 < 2 ? 2 : NS0);
  static constexpr int PRING = NS * STAGE;                // one pipeline's ring
  static constexpr int OBUF = NW * (HM ? 16 : 8) * D * 4;   // merge buffer (reuses the rings)
  static constexpr int RING = NP * PRING > OBUF ? NP * PRING : OBUF;
  static constexpr int BAR_OFF = RING;                    // [NP][full NS | empty NS] mbarriers
  static constexpr int OK_OFF = BAR_OFF + NP * 2 * NS * 8;  // [NP][NS] "tile is valid" flags, then a flag
  static constexpr int KB_OFF = OK_OFF + 128;             // QK accumulator seeds [HG][NB][4] f32x2
  static constexpr int ML_OFF = KB_OFF + HG * NB * 4 * 8; // per-warp m, l [NW][8][2] (HM: [NW][16][2])
  static constexpr int ML_BYTES = HM ? (NW + HG) * 16 * 8 : (NW + 2) * 16 * 4;
  static constexpr int PG_OFF = ML_OFF + ML_BYTES;        // + per-head (M, l); then [NP][64] page ids
  static constexpr int RC_OFF = PG_OFF + NP * 64 * 4;     // [NP][NS] releases counted per stage
  static constexpr int LI_OFF = RC_OFF + 16 * 4;          // [NP][NS] last tile issued into each stage
  // HM: q in MMA fragment order [HG][D/16][32 lanes] x 16 bytes, then the QK seeds
  // [HG][NB][8] f32x4 (rows r, r, r + 8, r + 8)
  static constexpr int QF_OFF = LI_OFF + 16 * 4;
  static constexpr int SD_OFF = QF_OFF + (HM ? HG * (D / 16) * 512 : 0);
  // HM: per warp, the f32 block scales of its 16-token slice, K [NB][16] then V [NB][16]
  static constexpr int SC_OFF = SD_OFF + (HM ? HG * NB * 128 : 0);
  static constexpr int SMEM = SC_OFF + (HM ? NW * 2 * NB * 16 * 4 : 0) + 1024;   // +1024: alignment
  static constexpr uint32_t K_TX = kT * KRB + (KQ ? kT * NB * 2 : 0);
  static constexpr uint32_t V_TX = kT * VRB + (VQ ? kT * NB * 2 : 0);
  static constexpr int QSTEPS = D / 16;                   // k16 steps of QK^T
  // 233472 bytes of shared memory per SM, 1024 of them reserved per resident CTA
  static_assert(!PACK || SMEM + 1024 <= 233472, "the four pipelines must fit one SM");
  static_assert(NP * NS <= 16, "stage flags");
  static_assert(!HM || SMEM <= 232448, "heads-on-M configuration exceeds shared memory");
};

// Shared-memory address of 16-byte chunk `chunk` of tile row `t` (rows as TMA wrote them).
template <int RB>
__device__ __forceinline__ uint32_t row_chunk(uint32_t base, int t, int chunk) {
  if constexpr (RB >= 128) {
    return base + (chunk >> 3) * (kT * 128) + t * 128 + (((chunk & 7) ^ (t & 7)) << 4);
  } else if constexpr (RB == 64) {
    return base + t * 64 + ((chunk ^ ((t >> 1) & 3)) << 4);
  } else {
    return base + t * 32 + ((chunk ^ ((t >> 2) & 1)) << 4);
  }
}

// Element of head_dim held by k-slot `k` (0..15) of QK^T step `s` for the K codec.
template <int KC>
__device__ __forceinline__ int qk_dim(int s, int k) {
  const int i = (k & 7) >> 1, e = k & 1, hi = k >> 3;
  if constexpr (KC == KVQ_CODEC_Q8_0) return 16 * s + 4 * i + 2 * hi + e;
  else if constexpr (KC == KVQ_CODEC_Q4S) return 32 * (s >> 1) + 8 * i + 2 * (s & 1) + hi + 4 * e;
  else return 16 * s + k;
}
// Element of head_dim held by row `row` (0..15) of PV M-tile `mt` for the V codec.
template <int VC>
__device__ __forceinline__ int pv_dim(int mt, int row) {
  const int b = mt >> 1, x = mt & 1, r = row & 7, top = row >> 3;
  if constexpr (VC == KVQ_CODEC_Q8_0) return 32 * b + 16 * top + 2 * r + x;
  else if constexpr (VC == KVQ_CODEC_Q4S) return 32 * b + 4 * r + 2 * x + top;
  else return 16 * mt + row;
}

// ---------------------------------------------------------------- split-K merge helpers

constexpr int kGroup = kMergeGroup;

// Counts this CTA's arrival on `counter` after its partial writes and tells whether it
// is the last of `expected` arrivals (all threads get the answer).  The last CTA sees
// every other CTA's writes.
__device__ __forceinline__ bool arrive_last(unsigned* counter, int expected, int tid, int nthreads,
                                            volatile int* flag, int32_t* status) {
  // bar.sync orders every thread's partial writes before thread 0's release-add at GPU
  // scope; the last CTA's acquire-add (and bar.sync) makes all of them visible to it.
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  if (tid == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    if (old >= (unsigned)expected) record_fault(status, KVQ_DEVICE_BAD_WORKSPACE);
    *flag = (old == (unsigned)expected - 1) ? 1 : 0;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
  return *flag != 0;
}

// Merges `count` split-K partials of each of `gcount` consecutive heads:
//   M = max_c m_c, l = sum_c 2^(m_c - M) l_c, O = sum_c 2^(m_c - M) O_c.
// Head h's partial c sits at ml[(h * stride + c) * 2] and o[(h * stride + c) * D].
// With `final` the normalized output O / l goes to out[h * D]; otherwise (M, l, O) go
// to out_ml[h * out_stride * 2] / out_o[h * out_stride * D].  Every thread of the CTA
// takes part (it contains a CTA barrier).
//
// Latency is what counts here (the last CTA of a split runs it after everything else):
// the items (head, 4 consecutive elements) are spread over the CTA's threads together
// with the partials, so that each thread loads at most kBatch partials, all at once (one
// L2 round trip); when several threads share an item, their running results meet in
// shared memory (`scratch`, 6 floats per thread) and one of them folds them in order.
template <int D, int NW>
__device__ void merge_partials(const float* ml, const float* o, long long stride, int count, int gcount,
                               bool final, float* out_ml, float* out_o, long long out_stride, float* out,
                               float* scratch) {
  constexpr int D4 = D / 4;
  constexpr int NT = NW * 32;
  constexpr int kBatch = 8;
  const int items = gcount * D4;
  int nsplit = NT / items;                        // threads per item
  if (nsplit > count) nsplit = count;
  if (nsplit < 1) nsplit = 1;
  const int per = (count + nsplit - 1) / nsplit;  // partials per thread
  // running (M, den, acc) of partials [c0, c1) of item `item`
  auto fold = [&](int item, int c0, int c1, float& M, float& den, float4& acc) {
    const int h = item / D4, col = item % D4;
    const float2* ml_h = reinterpret_cast<const float2*>(ml + h * stride * 2);
    const float4* o_h = reinterpret_cast<const float4*>(o + h * stride * D) + col;
    M = -INFINITY;
    den = 0.0f;
    acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int b0 = c0; b0 < c1; b0 += kBatch) {
      const int n = min(kBatch, c1 - b0);
      float2 mlv[kBatch];
      float4 v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (u < n) {
          mlv[u] = __ldcg(ml_h + b0 + u);
          v[u] = __ldcg(o_h + (long long)(b0 + u) * D4);
        }
      }
      float bm = M;
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (u < n) bm = fmaxf(bm, mlv[u].x);
      if (bm == -INFINITY) continue;
      const float f = fast_exp2(M - bm);   // 0 when M = -inf
      den *= f;
      acc.x *= f; acc.y *= f; acc.z *= f; acc.w *= f;
      M = bm;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (u < n && mlv[u].x != -INFINITY) {
          const float w = fast_exp2(mlv[u].x - M);
          den = fmaf(w, mlv[u].y, den);
          acc.x = fmaf(w, v[u].x, acc.x);
          acc.y = fmaf(w, v[u].y, acc.y);
          acc.z = fmaf(w, v[u].z, acc.z);
          acc.w = fmaf(w, v[u].w, acc.w);
        }
      }
    }
  };
  auto emit = [&](int item, float M, float den, float4 acc) {
    const int h = item / D4, col = item % D4;
    if (final) {
      const float inv = den > 0.0f ? 1.0f / den : 0.0f;
      reinterpret_cast<float4*>(out + h * D)[col] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      reinterpret_cast<float4*>(out_o + h * out_stride * D)[col] = acc;
      if (col == 0) reinterpret_cast<float2*>(out_ml + h * out_stride * 2)[0] = make_float2(M, den);
    }
  };
  // one (item, slice) per thread when the items are split (items * nsplit <= NT), else
  // every thread folds whole items in turn
  const int t = threadIdx.x;
  for (int it = t; it < items * nsplit; it += NT) {
    const int item = it % items, sg = it / items;
    float M, den;
    float4 acc;
    fold(item, sg * per, min(count, sg * per + per), M, den, acc);
    if (nsplit == 1) {
      emit(item, M, den, acc);
    } else {
      float* sc = scratch + it * 6;
      sc[0] = M; sc[1] = den; sc[2] = acc.x; sc[3] = acc.y; sc[4] = acc.z; sc[5] = acc.w;
    }
  }
  if (nsplit == 1) return;
  asm volatile("bar.sync 1, %0;" ::"r"(NT) : "memory");
  for (int item = t; item < items; item += NT) {
    float M = -INFINITY;
    for (int sg = 0; sg < nsplit; ++sg) M = fmaxf(M, scratch[(sg * items + item) * 6]);
    float den = 0.0f;
    float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (M != -INFINITY) {
      for (int sg = 0; sg < nsplit; ++sg) {
        const float* sc = scratch + (sg * items + item) * 6;
        if (sc[0] == -INFINITY) continue;
        const float w = fast_exp2(sc[0] - M);
        den = fmaf(w, sc[1], den);
        acc.x = fmaf(w, sc[2], acc.x);
        acc.y = fmaf(w, sc[3], acc.y);
        acc.z = fmaf(w, sc[4], acc.z);
        acc.w = fmaf(w, sc[5], acc.w);
      }
    }
    emit(item, M, den, acc);
  }
}

// Split-K combine (a8) after a CTA wrote its chunk partial.  Two levels, both done by
// whichever CTA arrives last (atomic counters in the workspace, returned to zero by that
// CTA):
//   group: the last of the <= kGroup chunks of a group merges their partials into a
//          group partial while the rest of the grid is still streaming;
//   unit:  the last group of a (sequence, KV head) merges the group partials into the
//          output.  A single group (up to 64 chunks form one) writes the output directly.
template <int D, int NW>
__device__ __forceinline__ void split_k_combine(const DecodeArgs& a, uint8_t* smem, volatile int* last_flag, int b,
                                                int kvh, int chunk, int nv, long long head0, int gcount) {
  const int tid = threadIdx.x, NWT = NW * 32;
  const long long unit = (long long)b * a.k.num_kv_heads + kvh;
  const int gsz = nv <= 4 * kGroup ? nv : kGroup;   // up to 64 partials: one level
  const int ng = (nv + gsz - 1) / gsz;
  const int g = chunk / gsz;
  const int g_first = g * gsz;
  const int g_count = min(gsz, nv - g_first);
  if (!arrive_last(a.counters + a.grp_counter_off + unit * a.n_groups + g, g_count, tid, NWT, last_flag,
                   a.k.status))
    return;
  // merge this group's chunk partials
  merge_partials<D, NW>(
      a.part_ml + (head0 * a.n_chunks + g_first) * 2, a.part_o + (head0 * a.n_chunks + g_first) * D,
      (long long)a.n_chunks, g_count, gcount, ng == 1,
      a.gpart_ml + (head0 * a.n_groups + g) * 2, a.gpart_o + (head0 * a.n_groups + g) * D,
      (long long)a.n_groups, a.out + head0 * D, reinterpret_cast<float*>(smem));
  if (tid == 0) a.counters[a.grp_counter_off + unit * a.n_groups + g] = 0u;
  if (ng == 1) {
    return;
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NWT) : "memory");   // group partial written before arriving
  if (!arrive_last(a.counters + unit, ng, tid, NWT, last_flag, a.k.status)) return;
  // the group partials were written by other CTAs before their arrivals
  merge_partials<D, NW>(a.gpart_ml + head0 * a.n_groups * 2, a.gpart_o + head0 * a.n_groups * D,
                        (long long)a.n_groups, ng, gcount, true, nullptr, nullptr, 0, a.out + head0 * D,
                        reinterpret_cast<float*>(smem));
  if (tid == 0) a.counters[unit] = 0u;
}

}  // namespace mma
}  // namespace kvq

#include "kvq_decode_hm.cuh"

namespace kvq {
namespace mma {

// ---------------------------------------------------------------- kernel

// Arrival on a per-sequence counter (release: the arriving CTA's reads of seq_lens come
// before it); returns the ticket.
__device__ __forceinline__ unsigned seq_arrive(unsigned* cnt) {
  unsigned old;
  asm volatile("atom.release.gpu.global.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(cnt) : "memory");
  return old;
}

template <int KC, int VC, int D, int GW, int HG, bool SOLO>
__device__ __forceinline__ void decode_cta(const CUtensorMap& tmk, const CUtensorMap& tmv, const DecodeArgs& a) {
  using C = Cfg<KC, VC, D, GW, HG, SOLO>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the 128-byte swizzle pattern
  // (offset from the array itself, so accesses through `smem` stay in the shared space)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Pipeline of this warp: its own ring of NS stages, barriers and stage flags.  The CTA's
  // pipelines take the tiles of "virtual chunks" vchunk = pipe * n_chunks + chunk
  // (pipe-major, so that the pipelines dealt one more tile than the rest spread over all
  // the CTAs of the unit: every SM gets the same number of tiles, to within one).
  const int pipe = warp / C::PW, pw = warp % C::PW;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sring = sbase + pipe * C::PRING;                 // this pipeline's ring
  uint8_t* const ring = smem + pipe * C::PRING;
  const uint32_t bar_full = sbase + C::BAR_OFF + pipe * 16 * C::NS;   // + 8*s
  const uint32_t bar_empty = bar_full + 8 * C::NS;
  float* ml_all = reinterpret_cast<float*>(smem + C::ML_OFF);
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + C::OK_OFF) + pipe * C::NS;
  const int vchunk = pipe * a.n_chunks + chunk;
  const int nvc = a.n_chunks * C::NP;
  const int G = a.group;         // query heads (virtual: head x query token) per KV head
  const int T = a.tokens;        // query tokens per sequence (1: plain decode)
  const int P = a.k.page_size;

  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  // Launched with programmatic stream serialization: nothing above reads memory an
  // earlier kernel may write; wait for that kernel here, and let the next one launch.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int32_t* pt = a.page_table + (long long)b * a.max_pages;
  // heads-on-M loop: this thread's q loads, in flight with the reads below
  HmQ<KC, D, HG, C::THREADS, C::HM> hmq;
  hmq.load(a, (long long)b * a.num_q_heads + (long long)kvh * G, G);
  // Page ids of this CTA's tiles, held by warp 0: lane i has tile pb + i in pg_lo and
  // tile pb + 32 + i in pg_hi.  The first 64 are read together with seq_lens (any
  // in-bounds table entry may be read; entries past the sequence are never used).
  auto load_page = [&](int tile) -> int {
    const long long pos0 = ((long long)vchunk + (long long)tile * nvc) * kT;
    return pos0 < (long long)a.max_pages * P ? __ldg(pt + pos0 / P) : -1;
  };
  int pg_lo = -1, pg_hi = -1, pb = 0;
  if (pw == 0) {
    pg_lo = load_page(lane);
    pg_hi = load_page(32 + lane);
  }
  // Fused append: the new token's K and V rows, read early by warp 0 (used only by the
  // CTA whose tile holds the token; the reads are in bounds for every CTA).
  constexpr int EPL = D / 32;
  float xk[EPL], xv[EPL];
  if (a.k_new != nullptr && pw == 0) {
    const long long row = (long long)b * a.k.num_kv_heads + kvh;
    load_row<EPL>(a.k_new + row * D, lane, xk);
    load_row<EPL>(a.v_new + row * D, lane, xv);
  }
  const long long cap = min((long long)a.max_pages * P, (long long)a.n_chunks * a.chunk_tokens);
  const bool fused = a.k_new != nullptr;
  const long long L_old = a.seq_lens[b];
  long long Lraw = fused ? L_old + 1 : L_old;
  const bool len_ok = L_old >= 0 && Lraw <= cap;   // else: fault, no append, no advance
  if (!len_ok) {
    if (tid == 0 && chunk == 0 && kvh == 0) {
      record_fault(a.k.status, KVQ_DEVICE_BAD_SEQ_LEN);
      record_fault(a.v.status, KVQ_DEVICE_BAD_SEQ_LEN);
    }
    Lraw = L_old < 0 ? 0 : cap;
  }
  const int L = (int)Lraw;
  // The sequence's 64-token tiles are dealt round-robin to the nvc pipelines of its
  // n_chunks CTAs: pipeline v takes tiles v, v + nvc, ... so that every pipeline streams
  // from all of the sequence's pages (evens out per-pipeline speed) and all finish together.
  const int NT = (L + kT - 1) / kT;                 // tiles of the sequence
  const int nv = min(a.n_chunks, NT);   // CTAs with work for this (b, kvh): pipeline 0 has a tile
  // Fused advance of seq_lens[b]: every CTA of the sequence takes one ticket on its
  // counter once all its threads have read seq_lens[b] (a CTA barrier, then a release
  // add), early in the kernel and off the tile producer's path; the holder of the last
  // ticket stores the new length and returns the counter to zero.  Nothing of it is left
  // for the end of the kernel.
  const bool adv = a.seq_lens_adv != nullptr;
  auto seq_ticket = [&]() {   // one thread per CTA, after a CTA barrier
    const unsigned total = gridDim.x * gridDim.y;
    const unsigned ticket = seq_arrive(a.seq_counters + b);
    if (ticket >= total) record_fault(a.k.status, KVQ_DEVICE_BAD_WORKSPACE);
    if (ticket == total - 1) {
      asm volatile("fence.acq_rel.gpu;" ::: "memory");   // after every counted arrival
      if (len_ok) a.seq_lens_adv[b] = (int32_t)(L_old + 1);
      a.seq_counters[b] = 0u;
    }
  };
  if (chunk >= nv) {
    if (C::LEAN && a.warp_records > 0) {
      // record mode: this CTA's records are empty (m = -inf), the merge skips them
      const long long rec0 = ((long long)b * gridDim.y + kvh) * a.warp_records + (long long)chunk * C::NW;
      for (int i = tid; i < C::NW * 2; i += C::THREADS)
        reinterpret_cast<float4*>(a.part_ml + (rec0 + i / 2) * 8)[i & 1] = make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
    } else if (C::HM && a.chunk_merge) {
      // chunk-merge mode: this CTA's partial is empty (m = -inf), the merge skips it
      const long long h0 = (long long)b * a.num_q_heads + (long long)kvh * G;
      for (int v = tid; v < G; v += C::THREADS)
        reinterpret_cast<float2*>(a.part_ml)[(h0 + v) * a.n_chunks + chunk] = make_float2(-INFINITY, 0.0f);
    } else if (L == 0 && chunk == 0) {  // empty sequence: its heads' outputs are zero
      const long long h0 = (long long)b * a.num_q_heads + (long long)kvh * G;
      for (int idx = tid; idx < G * D; idx += C::THREADS) a.out[h0 * D + idx] = 0.0f;
    }
    if (adv && !(C::LEAN && a.warp_records > 0)) {
      __syncthreads();   // every thread has read seq_lens
      if (tid == 0) seq_ticket();
    }
    return;
  }
  const int n_tiles = vchunk < NT ? (NT - vchunk + nvc - 1) / nvc : 0;   // this pipeline's

  if (pw == 0 && lane == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, C::PW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // lean loop: the page ids of the pipeline's first 64 tiles and the release counters live
  // in shared memory, where whichever warp refills a stage finds them
  int* const pgs = reinterpret_cast<int*>(smem + C::PG_OFF) + pipe * 64;
  unsigned* const rcnt = reinterpret_cast<unsigned*>(smem + C::RC_OFF) + pipe * C::NS;
  volatile int* const last_issued = reinterpret_cast<volatile int*>(smem + C::LI_OFF) + pipe * C::NS;
  if (pw == 0 && lane < C::NS) last_issued[lane] = -1;
  if ((C::LEAN || C::HM) && pw == 0) {
    pgs[lane] = pg_lo;
    pgs[32 + lane] = pg_hi;
    if (lane < C::NS) rcnt[lane] = 0u;
  }
  __syncthreads();   // also: every thread has read seq_lens

  // ------------------------------------------------------------ tile producer
  // Lane 0 of the pipeline's first warp issues its copies: the first NS tiles up front,
  // then tile k + NS into stage k % NS as soon as every warp of the pipeline has released
  // tile k.
  // Copies of the pipeline's local tile `tile` (into stage tile % NS), which is the sequence's
  // 64-token tile g.
  auto issue_at = [&](int tile, int g, int page) {
    const int s = tile % C::NS;
    // fault injection (tests of the timeout path): the first pipeline never issues this
    // tile, neither its copies nor an arrival, so its consumers' bounded waits run out on a
    // stage with nothing in flight
    if (vchunk == 0 && tile == a.skip_tile) return;
    last_issued[s] = tile;
    const int pos0 = g * kT;
    const int row0 = pos0 % P;
    const uint32_t full = bar_full + 8 * s;
    // the flag is published to the warps by the mbarrier phase that completes below
    const bool ok = page >= 0 && page < a.k.num_pages && page < a.v.num_pages;
    stage_ok[s] = ok ? 1 : 0;
    if (!ok) {
      record_fault(a.k.status, KVQ_DEVICE_BAD_PAGE);
      record_fault(a.v.status, KVQ_DEVICE_BAD_PAGE);
      mbar_arrive(full);
      return;
    }
    mbar_expect_tx(full, C::K_TX + C::V_TX);
    const uint32_t st = sring + s * C::STAGE;
    const uint64_t pol = evict_first_policy();
#pragma unroll
    for (int seg = 0; seg < (C::KRB + 127) / 128; ++seg)
      tma_load_4d_ef(st + seg * kT * 128, &tmk, seg * 128, row0, kvh, page, full, pol);
    const uint32_t vst = st + C::V_OFF;
#pragma unroll
    for (int seg = 0; seg < (C::VRB + 127) / 128; ++seg)
      tma_load_4d_ef(vst + seg * kT * 128, &tmv, seg * 128, row0, kvh, page, full, pol);
    if constexpr (C::KQ) {
      const uint8_t* src = a.k.buf + ((long long)page * a.k.num_kv_heads + kvh) * a.k.slab_bytes +
                           (long long)P * C::KRB + (long long)row0 * C::NB * 2;
      bulk_load_ef(st + C::KSC_OFF, src, kT * C::NB * 2, full, pol);
    }
    if constexpr (C::VQ) {
      const uint8_t* src = a.v.buf + ((long long)page * a.v.num_kv_heads + kvh) * a.v.slab_bytes +
                           (long long)P * C::VRB + (long long)row0 * C::NB * 2;
      bulk_load_ef(st + C::VSC_OFF, src, kT * C::NB * 2, full, pol);
    }
  };
  // local tile t is the sequence's tile vchunk + t * nvc
  auto issue_tile = [&](int tile, int page) { issue_at(tile, vchunk + tile * nvc, page); };
  // Page of tile t (t >= pb, nondecreasing over calls), by all of the producer warp.  Crossing a
  // 32-tile boundary shifts the window and starts the loads for the batch after next,
  // 32 tiles before they are needed.
  auto page_of = [&](int t) -> int {
    while (t >= pb + 32) {
      pg_lo = pg_hi;
      pb += 32;
      pg_hi = load_page(pb + 32 + lane);
    }
    return __shfl_sync(0xffffffffu, pg_lo, t - pb);
  };
  // Fused append: the CTA holding the new token's tile (its last) encodes the token's K
  // and V rows with warp 0 before that tile's copies are issued; the proxy fence orders
  // the rows' generic-proxy stores before the bulk-tensor reads.
  bool need_enc = fused && len_ok && vchunk == (NT - 1) % nvc;
  auto encode_new = [&]() {   // by all of the producer warp; the token lies in its pipeline's last tile
    const int t = n_tiles - 1;   // read without moving page_of's window
    const int lo = __shfl_sync(0xffffffffu, pg_lo, (t - pb) & 31);
    const int hi = __shfl_sync(0xffffffffu, pg_hi, (t - pb) & 31);
    const int page = t < pb + 32 ? lo : t < pb + 64 ? hi : load_page(t);
    if (page >= 0 && page < a.k.num_pages && page < a.v.num_pages) {   // else the tile faults
      const int r = (int)(L_old % P);
      store_row<KC, EPL>(a.k, page, r, kvh, xk);
      store_row<VC, EPL>(a.v, page, r, kvh, xv);
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncwarp();
    need_enc = false;
  };
  if (pw == 0) {
    for (int tile = 0; tile < n_tiles && tile < C::NS; ++tile) {
      if (need_enc && tile == n_tiles - 1) encode_new();
      const int page = page_of(tile);
      if (lane == 0) issue_tile(tile, page);
    }
    __syncwarp();
    if (need_enc) encode_new();   // its tile comes later, from the refill path
  }

  if constexpr (C::HM) {
    // ---------------------------------------------------------- heads-on-M loop
    if (hm_body<KC, VC, D, GW, HG>(a, smem, b, kvh, chunk, pipe, pw, warp, lane, tid, vchunk, nvc, n_tiles, L, nv,
                                   sring, bar_full, bar_empty, stage_ok, pgs, rcnt, last_issued, issue_tile,
                                   load_page, adv, seq_ticket, hmq))
      split_k_combine<D, C::NW>(a, smem, reinterpret_cast<volatile int*>(smem + C::OK_OFF) + 16, b, kvh, chunk, nv,
                                (long long)b * a.num_q_heads + (long long)kvh * G, G < 16 * HG ? G : 16 * HG);
  } else {   // tokens-on-M loop
  // ------------------------------------------------------------ compute warps
  const int hg = pw >> 2;            // head group
  const int ws = pw & 3;             // 16-token slice of every tile
  const int r = lane >> 2, i4 = lane & 3;
  const int t0 = ws * 16;

  // q fragments (B operand of QK^T): column r, k-slots {2i, 2i+1} and {2i+8, 2i+9}.
  // With at most 4 heads per warp, columns 4..7 repeat heads 0..3, so that after the
  // transpose of p every PV column (head, hi|lo) finds its head's p in its own lane.
  uint32_t qf[C::QSTEPS][2];
  {
    const int h = hg * GW + (GW <= 4 ? (r & 3) : r);
    const bool hv = h < G;
    const __nv_bfloat16* qrow = a.q + ((long long)b * a.num_q_heads + (long long)kvh * G + (hv ? h : 0)) * D;
#pragma unroll
    for (int s = 0; s < C::QSTEPS; ++s) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const float x0 = hv ? __bfloat162float(qrow[qk_dim<KC>(s, 8 * half + 2 * i4)]) : 0.0f;
        const float x1 = hv ? __bfloat162float(qrow[qk_dim<KC>(s, 8 * half + 2 * i4 + 1)]) : 0.0f;
        qf[s][half] = pack2<C::KBF>(x0, x1);
      }
    }
  }

  // Per block: -bias * sum_j q[h, j] for the S columns 2i, 2i+1 of this lane (zero for
  // 16-bit K), the seed of the block's QK accumulator.  Summed from the f16 values the
  // MMA multiplies; lanes r = n hold column n's B operand, so column n's sum comes from
  // lane 4n after a quad reduction.
  // Kept in shared memory ([head group][block][i4], float2): every lane of a head group
  // with the same i4 needs the same pair.
  float2* kbs = reinterpret_cast<float2*>(smem + C::KB_OFF);
  float2 kbr[C::NB];   // the same seeds in registers (lean loop)
#pragma unroll
  for (int bb = 0; bb < C::NB; ++bb) {
    float part = 0.0f;
    if constexpr (C::KQ) {
#pragma unroll
      for (int st = 2 * bb; st < 2 * bb + 2; ++st)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const float2 f = unpack2<false>(qf[st][half]);
          part += f.x + f.y;
        }
      part += __shfl_xor_sync(0xffffffffu, part, 1);
      part += __shfl_xor_sync(0xffffffffu, part, 2);
    }
    const float bias = KC == KVQ_CODEC_Q4S ? kBias4K : kBias8;
    const float k0 = -bias * __shfl_sync(0xffffffffu, part, 4 * (2 * i4));
    const float k1 = -bias * __shfl_sync(0xffffffffu, part, 4 * (2 * i4 + 1));
    if (!C::LEAN && pipe == 0 && ws == 0 && r == 0) kbs[(hg * C::NB + bb) * 4 + i4] = make_float2(k0, k1);
    kbr[bb] = make_float2(k0, k1);
  }
  if constexpr (!C::LEAN) asm volatile("bar.sync 1, %0;" ::"r"(C::THREADS) : "memory");   // seeds in smem
  // Fused advance outside record mode (there the merge kernel stores the new length): the
  // last warp takes the CTA's ticket, after every CTA-wide barrier before the tile loop,
  // so that its wait holds up no other warp.
  if (adv && !(C::LEAN && a.warp_records > 0) && warp == C::NW - 1 && lane == 0) seq_ticket();

  float o[C::QSTEPS][C::NPV][4];   // O^T accumulators: D/16 M-tiles x NPV n-tiles
#pragma unroll
  for (int mt = 0; mt < C::QSTEPS; ++mt)
#pragma unroll
    for (int n = 0; n < C::NPV; ++n)
#pragma unroll
      for (int k = 0; k < 4; ++k) o[mt][n][k] = 0.0f;
  // reference max (warp-uniform) and this lane's partial sum for QK columns 2*i4, 2*i4+1
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
  // softmax scale in log2 units; 4-bit K fragments carry q/8
  const float qk_mul = a.qk_scale_log2 * (KC == KVQ_CODEC_Q4S ? kScale4K : 1.0f);
  int E = -100;                                                 // running V-scale exponent bound
  bool timed_out = false;
  const int wlim = a.wait_limit;   // tries of mbarrier.try_wait before a wait gives up

  if constexpr (C::LEAN) {
    // ---------------------------------------------------------- lean tile loop
    // Warps of at most 4 heads (one 8-column MMA carries hi and lo parts of P).  Against
    // the general loop below: the stage index and phase advance incrementally; a slice
    // whose 16 tokens are all valid (every slice but a sequence's last) skips all
    // masking; the QK seeds stay in registers; and the V-scaled P of each head is formed
    // once per (token, block): lane (r, i) with r < 4 forms the hi and lo parts of tokens
    // 2i, 2i + 1 and its partner lane (r + 4, i) those of tokens 2i + 8, 2i + 9, and one
    // shuffle gives each its missing half (the hi lane needs the partner's hi, the lo
    // lane the partner's lo).
    const int mi = lane >> 3, mr = lane & 7;
    const bool hi_lane = r < 4;
    const int tp = hi_lane ? 2 * i4 : 2 * i4 + 8;   // this lane's two P tokens
    int s = 0;
    uint32_t ph = 0u;
    for (int tile = 0; tile < n_tiles; ++tile) {
      if (!mbar_wait_warp(bar_full + 8 * s, ph, wlim)) {
        timed_out = true;
        break;
      }
      const int pos_w = (vchunk + tile * nvc) * kT + t0;
      const int n_valid = stage_ok[s] != 0 ? max(0, min(16, L - pos_w)) : 0;
      if (n_valid > 0) {
        const bool causal = T > 1 && pos_w + 16 > L - T + 1;
        const bool slow = n_valid < 16 || causal;   // warp-uniform
        const uint32_t st = sring + s * C::STAGE;
        const uint32_t kst = st, vst = st + C::V_OFF;
        const uint8_t* ksc = ring + s * C::STAGE + C::KSC_OFF;
        const uint8_t* vsc = ring + s * C::STAGE + C::VSC_OFF;

        // ---------------- QK^T: S[tok r / r+8][heads 2i, 2i+1] (log2 units after scaling)
        float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if constexpr (C::KQ) {
          float dk[2][C::NB];
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            uint32_t w[C::NB / 2];
            load_scale_words<C::NB>(ksc, t0 + r + 8 * rr, w);
#pragma unroll
            for (int k = 0; k < C::NB / 2; ++k) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
              dk[rr][2 * k] = f.x;
              dk[rr][2 * k + 1] = f.y;
            }
          }
          if constexpr (KC == KVQ_CODEC_Q8_0) {
#pragma unroll
            for (int bb = 0; bb < C::NB; ++bb) {
              uint32_t x0, x1, x2, x3;
              ldsm_x4(row_chunk<C::KRB>(kst, t0 + (mi & 1) * 8 + mr, 2 * bb + (mi >> 1)), x0, x1, x2, x3);
              x0 ^= 0x80808080u; x1 ^= 0x80808080u; x2 ^= 0x80808080u; x3 ^= 0x80808080u;
              float cb[4] = {kbr[bb].x, kbr[bb].y, kbr[bb].x, kbr[bb].y};
              uint32_t af[4];
              af[0] = i8pair_raw(x0, 0x4140); af[1] = i8pair_raw(x1, 0x4140);
              af[2] = i8pair_raw(x0, 0x4342); af[3] = i8pair_raw(x1, 0x4342);
              mma16816<false>(cb, af, qf[2 * bb][0], qf[2 * bb][1]);
              af[0] = i8pair_raw(x2, 0x4140); af[1] = i8pair_raw(x3, 0x4140);
              af[2] = i8pair_raw(x2, 0x4342); af[3] = i8pair_raw(x3, 0x4342);
              mma16816<false>(cb, af, qf[2 * bb + 1][0], qf[2 * bb + 1][1]);
              sc[0] = fmaf(dk[0][bb], cb[0], sc[0]);
              sc[1] = fmaf(dk[0][bb], cb[1], sc[1]);
              sc[2] = fmaf(dk[1][bb], cb[2], sc[2]);
              sc[3] = fmaf(dk[1][bb], cb[3], sc[3]);
            }
          } else {  // q4s: one ldmatrix.x4 covers two blocks
#pragma unroll
            for (int bb = 0; bb < C::NB; bb += 2) {
              uint32_t x[4];
              ldsm_x4(row_chunk<C::KRB>(kst, t0 + (mi & 1) * 8 + mr, bb + (mi >> 1)), x[0], x[1], x[2], x[3]);
#pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t ra = x[2 * h2], rb = x[2 * h2 + 1];  // rows r and r+8 of block bb+h2
                float cb[4] = {kbr[bb + h2].x, kbr[bb + h2].y, kbr[bb + h2].x, kbr[bb + h2].y};
                uint32_t af[4];
                af[0] = u4pair_half(ra << 4); af[1] = u4pair_half(rb << 4);
                af[2] = u4pair_half(ra); af[3] = u4pair_half(rb);
                mma16816<false>(cb, af, qf[2 * (bb + h2)][0], qf[2 * (bb + h2)][1]);
                af[0] = u4pair_half(ra >> 4); af[1] = u4pair_half(rb >> 4);
                af[2] = u4pair_half(ra >> 8); af[3] = u4pair_half(rb >> 8);
                mma16816<false>(cb, af, qf[2 * (bb + h2) + 1][0], qf[2 * (bb + h2) + 1][1]);
                sc[0] = fmaf(dk[0][bb + h2], cb[0], sc[0]);
                sc[1] = fmaf(dk[0][bb + h2], cb[1], sc[1]);
                sc[2] = fmaf(dk[1][bb + h2], cb[2], sc[2]);
                sc[3] = fmaf(dk[1][bb + h2], cb[3], sc[3]);
              }
            }
          }
        } else {  // 16-bit K: natural k order, one ldmatrix.x4 per k16 step
#pragma unroll
          for (int ks = 0; ks < C::QSTEPS; ++ks) {
            uint32_t af[4];
            ldsm_x4(row_chunk<C::KRB>(kst, t0 + (mi & 1) * 8 + mr, 2 * ks + (mi >> 1)), af[0], af[1], af[2], af[3]);
            mma16816<C::KBF>(sc, af, qf[ks][0], qf[ks][1]);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) sc[k] *= qk_mul;
        if (slow) {
          if (r >= n_valid) { sc[0] = -INFINITY; sc[1] = -INFINITY; }
          if (r + 8 >= n_valid) { sc[2] = -INFINITY; sc[3] = -INFINITY; }
          if (causal) {
            // virtual head v = head * T + i sees the positions below L - T + 1 + i
            const int cA = 2 * i4, cB = 2 * i4 + 1;
            const int vA = cA & 3, vB = cB & 3;
            const int limA = L - T + 1 + vA % T, limB = L - T + 1 + vB % T;
            if (pos_w + r >= limA) sc[0] = -INFINITY;
            if (pos_w + r >= limB) sc[1] = -INFINITY;
            if (pos_w + r + 8 >= limA) sc[2] = -INFINITY;
            if (pos_w + r + 8 >= limB) sc[3] = -INFINITY;
          }
        }

        // ---------------- V scales of this lane's two P tokens (all blocks), their bound
        uint32_t dw[C::VQ ? C::NB : 1];   // tokens tp (words 0..NB/2-1) and tp+1 (the rest)
        int ex_lane = 0;   // every scale of this lane's tokens is < 2^ex_lane
        if constexpr (C::VQ) {
          const uint8_t* p2 = vsc + (t0 + tp) * C::NB * 2;
          if constexpr (C::NB == 4) {
            const uint4 v = *reinterpret_cast<const uint4*>(p2);
            dw[0] = v.x; dw[1] = v.y; dw[2] = v.z; dw[3] = v.w;
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(p2);
            dw[0] = v.x; dw[1] = v.y;
          }
          if (slow) {
#pragma unroll
            for (int k = 0; k < C::NB; ++k)
              if (tp + (2 * k >= C::NB ? 1 : 0) >= n_valid) dw[k] = 0u;
          }
          uint32_t mx = dw[0];
#pragma unroll
          for (int k = 1; k < C::NB; ++k) mx = __vmaxu2(mx, dw[k]);
          const uint32_t hmax = max(mx & 0xffffu, mx >> 16);   // scales are >= 0: bits order as values
          const int e = (int)(hmax >> 10);
          ex_lane = hmax ? max(e, 1) - 14 : -127;
        }

        // ---------------- lazy online softmax over the warp's 16 tokens (columns = heads)
        const float lm0 = fmaxf(sc[0], sc[2]), lm1 = fmaxf(sc[1], sc[3]);
        const bool over = (lm0 > m0 + kLazy) || (lm1 > m1 + kLazy) || (ex_lane > E);
        if (__any_sync(0xffffffffu, over)) {
          float mx0 = lm0, mx1 = lm1;
          int ex = ex_lane;
#pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          // the scale bound over all 16 tokens: lanes 0..15 hold tokens 0..7, 16..31 tokens 8..15
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) ex = max(ex, __shfl_xor_sync(0xffffffffu, ex, off));
          const int E_new = max(E, ex);
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const float e2 = __uint_as_float((uint32_t)(127 + E - E_new) << 23);  // 2^(E - E_new)
          float f0 = (mn0 == -INFINITY) ? 1.0f : fast_exp2(m0 - mn0);
          float f1 = (mn1 == -INFINITY) ? 1.0f : fast_exp2(m1 - mn1);
          l0 *= f0;
          l1 *= f1;
          f0 *= e2;
          f1 *= e2;
#pragma unroll
          for (int mt = 0; mt < C::QSTEPS; ++mt) {
            o[mt][0][0] *= f0; o[mt][0][1] *= f1; o[mt][0][2] *= f0; o[mt][0][3] *= f1;
          }
          m0 = mn0;
          m1 = mn1;
          E = E_new;
        }
        // m0, m1 are finite here unless a causal limit masked a column everywhere so far
        float p0 = fast_exp2(sc[0] - m0);
        float p1 = fast_exp2(sc[1] - m1);
        float p2 = fast_exp2(sc[2] - m0);
        float p3 = fast_exp2(sc[3] - m1);
        if (causal) {
          if (sc[0] == -INFINITY) p0 = 0.0f;
          if (sc[1] == -INFINITY) p1 = 0.0f;
          if (sc[2] == -INFINITY) p2 = 0.0f;
          if (sc[3] == -INFINITY) p3 = 0.0f;
        }
        l0 += p0 + p2;
        l1 += p1 + p3;

        // ---------------- transpose p to the PV B layout (fp32 as two 16-bit halves):
        // lane (r, i) receives p[tok 2i, 2i+1, 2i+8, 2i+9][column r] and keeps its pair
        float pa, pb;
        {
          const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
          const uint32_t u2 = __float_as_uint(p2), u3 = __float_as_uint(p3);
          const uint32_t ah = movtrans(__byte_perm(u0, u1, 0x7632)), al = movtrans(__byte_perm(u0, u1, 0x5410));
          const uint32_t bh = movtrans(__byte_perm(u2, u3, 0x7632)), bl = movtrans(__byte_perm(u2, u3, 0x5410));
          const uint32_t xl = hi_lane ? al : bl, xh = hi_lane ? ah : bh;
          pa = __uint_as_float(__byte_perm(xl, xh, 0x5410));
          pb = __uint_as_float(__byte_perm(xl, xh, 0x7632));
        }
        const float pscale = __uint_as_float((uint32_t)(127 + kPScale - E) << 23);  // 2^(kPScale - E)
        pa *= pscale;
        pb *= pscale;
        // (hi, lo) parts of (x0, x1) for this lane's tokens -> the B registers of its column
        auto b_regs = [&](float x0, float x1, uint32_t& b0, uint32_t& b1) {
          const uint32_t hi = pack2<C::VBF>(x0, x1);
          float y0, y1;
          add_k_times<C::VBF>(hi, C::VBF ? 0xBF80 : 0xBC00, x0, x1, y0, y1);
          const uint32_t lo = pack2<C::VBF>(y0, y1);
          const uint32_t recv = __shfl_xor_sync(0xffffffffu, hi_lane ? lo : hi, 16);
          b0 = hi_lane ? hi : recv;
          b1 = hi_lane ? recv : lo;
        };

        // ---------------- PV
        if constexpr (C::VQ) {
          uint32_t vq4[4];   // q4s: one ldmatrix.x4 covers blocks bb and bb + 1 (bb even)
#pragma unroll
          for (int bb = 0; bb < C::NB; ++bb) {
            const uint32_t wa = dw[bb >> 1], wb = dw[C::NB / 2 + (bb >> 1)];
            const float da = __half2float(__ushort_as_half((unsigned short)(wa >> (16 * (bb & 1)))));
            const float db = __half2float(__ushort_as_half((unsigned short)(wb >> (16 * (bb & 1)))));
            uint32_t b0, b1;
            b_regs(pa * da, pb * db, b0, b1);
            if constexpr (VC == KVQ_CODEC_Q8_0) {
              uint32_t y0, y1, y2, y3;
              // matrices: (tok 0-7, chunk 2b), (tok 0-7, chunk 2b+1), (tok 8-15, 2b), (tok 8-15, 2b+1)
              ldsm_x4_t(row_chunk<C::VRB>(vst, t0 + (mi >> 1) * 8 + mr, 2 * bb + (mi & 1)), y0, y1, y2, y3);
              y0 ^= 0x80808080u; y1 ^= 0x80808080u; y2 ^= 0x80808080u; y3 ^= 0x80808080u;
              uint32_t ae[4] = {i8pair_raw(y0, 0x4240), i8pair_raw(y1, 0x4240), i8pair_raw(y2, 0x4240),
                                i8pair_raw(y3, 0x4240)};
              uint32_t ao[4] = {i8pair_raw(y0, 0x4341), i8pair_raw(y1, 0x4341), i8pair_raw(y2, 0x4341),
                                i8pair_raw(y3, 0x4341)};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                ae[k] = hsub2_u32(ae[k], 0x64806480u);
                ao[k] = hsub2_u32(ao[k], 0x64806480u);
              }
              mma16816<false>(o[2 * bb][0], ae, b0, b1);
              mma16816<false>(o[2 * bb + 1][0], ao, b0, b1);
            } else {  // q4s: matrices (tok 0-7, chunk b), (tok 8-15, chunk b) for this block
              if ((bb & 1) == 0)
                ldsm_x4_t(row_chunk<C::VRB>(vst, t0 + (mi & 1) * 8 + mr, bb + (mi >> 1)), vq4[0], vq4[1], vq4[2], vq4[3]);
              const uint32_t ya = (bb & 1) ? vq4[2] : vq4[0], yb = (bb & 1) ? vq4[3] : vq4[1];
              const uint32_t ya8 = ya >> 8, yb8 = yb >> 8;
              const uint32_t a01[4] = {hsub2_u32(u4pair_raw(ya), 0x64086408u),
                                       hfma2_u32(u4pair_hi_raw(ya), kSixteenth2, kMinus72x2),
                                       hsub2_u32(u4pair_raw(yb), 0x64086408u),
                                       hfma2_u32(u4pair_hi_raw(yb), kSixteenth2, kMinus72x2)};
              const uint32_t a23[4] = {hsub2_u32(u4pair_raw(ya8), 0x64086408u),
                                       hfma2_u32(u4pair_hi_raw(ya8), kSixteenth2, kMinus72x2),
                                       hsub2_u32(u4pair_raw(yb8), 0x64086408u),
                                       hfma2_u32(u4pair_hi_raw(yb8), kSixteenth2, kMinus72x2)};
              mma16816<false>(o[2 * bb][0], a01, b0, b1);
              mma16816<false>(o[2 * bb + 1][0], a23, b0, b1);
            }
          }
        } else {
          // 16-bit V: one B operand for every M-tile; in a partial slice zero the A lanes of
          // tokens past the end (their rows may hold anything)
          uint32_t b0, b1;
          b_regs(pa, pb, b0, b1);
          uint32_t kmask_lo = 0xffffffffu, kmask_hi = 0xffffffffu;
          if (slow) {
            kmask_lo = (2 * i4 < n_valid ? 0x0000ffffu : 0u) | (2 * i4 + 1 < n_valid ? 0xffff0000u : 0u);
            kmask_hi = (2 * i4 + 8 < n_valid ? 0x0000ffffu : 0u) | (2 * i4 + 9 < n_valid ? 0xffff0000u : 0u);
          }
#pragma unroll
          for (int mt = 0; mt < C::QSTEPS; ++mt) {
            uint32_t af[4];
            ldsm_x4_t(row_chunk<C::VRB>(vst, t0 + (mi >> 1) * 8 + mr, 2 * mt + (mi & 1)), af[0], af[1], af[2], af[3]);
            if (slow) { af[0] &= kmask_lo; af[1] &= kmask_lo; af[2] &= kmask_hi; af[3] &= kmask_hi; }
            mma16816<C::VBF>(o[mt][0], af, b0, b1);
          }
        }
      }
      __syncwarp();
      // Release the stage; the warp that releases it last (counted in shared memory)
      // refills it at once, so that no warp waits for the others and a stage is never
      // left empty while its refiller finishes other work.
      uint32_t last = 0u;
      if (lane == 0) {
        mbar_arrive(bar_empty + 8 * s);
        last = atomicAdd(rcnt + s, 1u) == (unsigned)(C::PW - 1) ? 1u : 0u;
        if (last) atomicExch(rcnt + s, 0u);
      }
      last = __shfl_sync(0xffffffffu, last, 0);
      if (last && tile + C::NS < n_tiles) {
        if (!mbar_wait_warp(bar_empty + 8 * s, ph, wlim)) {   // every release is in: no wait
          timed_out = true;
          break;
        }
        const int t2 = tile + C::NS;
        const int page = t2 < 64 ? pgs[t2] : load_page(t2);
        if (lane == 0) issue_tile(t2, page);
        __syncwarp();
      }
      if (++s == C::NS) {
        s = 0;
        ph ^= 1u;
      }
    }
  } else {
    for (int tile = 0; tile < n_tiles; ++tile) {
      const int s = tile % C::NS;
      if (!mbar_wait_warp(bar_full + 8 * s, (tile / C::NS) & 1, wlim)) {
        timed_out = true;
        break;
      }
      const int pos_w = (vchunk + tile * nvc) * kT + t0;
      const bool tile_ok = stage_ok[s] != 0;
      const int n_valid = tile_ok ? max(0, min(16, L - pos_w)) : 0;
      if (n_valid > 0) {
        const bool partial = n_valid < 16;
        const uint32_t st = sring + s * C::STAGE;
        const uint32_t kst = st, vst = st + C::V_OFF;
        const uint8_t* ksc = ring + s * C::STAGE + C::KSC_OFF;
        const uint8_t* vsc = ring + s * C::STAGE + C::VSC_OFF;
        const int mi = lane >> 3, mr = lane & 7;

        // ---------------- QK^T: S[tok r / r+8][heads 2i, 2i+1] (log2 units after scaling)
        float sc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if constexpr (C::KQ) {
          // block scales of rows r and r+8
          float dk[2][C::NB];
  #pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            uint32_t w[C::NB / 2];
            load_scale_words<C::NB>(ksc, t0 + r + 8 * rr, w);
  #pragma unroll
            for (int k = 0; k < C::NB / 2; ++k) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
              dk[rr][2 * k] = f.x;
              dk[rr][2 * k + 1] = f.y;
            }
          }
          if constexpr (KC == KVQ_CODEC_Q8_0) {
  #pragma unroll
            for (int bb = 0; bb < C::NB; ++bb) {
              uint32_t x0, x1, x2, x3;
              ldsm_x4(row_chunk<C::KRB>(kst, t0 + (mi & 1) * 8 + mr, 2 * bb + (mi >> 1)), x0, x1, x2, x3);
              x0 ^= 0x80808080u; x1 ^= 0x80808080u; x2 ^= 0x80808080u; x3 ^= 0x80808080u;
              // accumulator seeded with -1152 * sum(q) of the block: removes the code offset
              const float2 kb = kbs[(hg * C::NB + bb) * 4 + i4];
              float cb[4] = {kb.x, kb.y, kb.x, kb.y};
              uint32_t af[4];
              af[0] = i8pair_raw(x0, 0x4140); af[1] = i8pair_raw(x1, 0x4140);
              af[2] = i8pair_raw(x0, 0x4342); af[3] = i8pair_raw(x1, 0x4342);
              mma16816<false>(cb, af, qf[2 * bb][0], qf[2 * bb][1]);
              af[0] = i8pair_raw(x2, 0x4140); af[1] = i8pair_raw(x3, 0x4140);
              af[2] = i8pair_raw(x2, 0x4342); af[3] = i8pair_raw(x3, 0x4342);
              mma16816<false>(cb, af, qf[2 * bb + 1][0], qf[2 * bb + 1][1]);
              sc[0] = fmaf(dk[0][bb], cb[0], sc[0]);
              sc[1] = fmaf(dk[0][bb], cb[1], sc[1]);
              sc[2] = fmaf(dk[1][bb], cb[2], sc[2]);
              sc[3] = fmaf(dk[1][bb], cb[3], sc[3]);
            }
          } else {  // q4s: one ldmatrix.x4 covers two blocks
  #pragma unroll
            for (int bb = 0; bb < C::NB; bb += 2) {
              uint32_t x[4];
              ldsm_x4(row_chunk<C::KRB>(kst, t0 + (mi & 1) * 8 + mr, bb + (mi >> 1)), x[0], x[1], x[2], x[3]);
  #pragma unroll
              for (int h2 = 0; h2 < 2; ++h2) {
                const uint32_t ra = x[2 * h2], rb = x[2 * h2 + 1];  // rows r and r+8 of block bb+h2
                const float2 kb = kbs[(hg * C::NB + bb + h2) * 4 + i4];
                float cb[4] = {kb.x, kb.y, kb.x, kb.y};
                uint32_t af[4];
                af[0] = u4pair_half(ra << 4); af[1] = u4pair_half(rb << 4);
                af[2] = u4pair_half(ra); af[3] = u4pair_half(rb);
                mma16816<false>(cb, af, qf[2 * (bb + h2)][0], qf[2 * (bb + h2)][1]);
                af[0] = u4pair_half(ra >> 4); af[1] = u4pair_half(rb >> 4);
                af[2] = u4pair_half(ra >> 8); af[3] = u4pair_half(rb >> 8);
                mma16816<false>(cb, af, qf[2 * (bb + h2) + 1][0], qf[2 * (bb + h2) + 1][1]);
                sc[0] = fmaf(dk[0][bb + h2], cb[0], sc[0]);
                sc[1] = fmaf(dk[0][bb + h2], cb[1], sc[1]);
                sc[2] = fmaf(dk[1][bb + h2], cb[2], sc[2]);
                sc[3] = fmaf(dk[1][bb + h2], cb[3], sc[3]);
              }
            }
          }
        } else {  // 16-bit K: natural k order, one ldmatrix.x4 per k16 step
  #pragma unroll
          for (int ks = 0; ks < C::QSTEPS; ++ks) {
            uint32_t af[4];
            ldsm_x4(row_chunk<C::KRB>(kst, t0 + (mi & 1) * 8 + mr, 2 * ks + (mi >> 1)), af[0], af[1], af[2], af[3]);
            mma16816<C::KBF>(sc, af, qf[ks][0], qf[ks][1]);
          }
        }
  #pragma unroll
        for (int k = 0; k < 4; ++k) sc[k] *= qk_mul;
        if (partial) {
          if (r >= n_valid) { sc[0] = -INFINITY; sc[1] = -INFINITY; }
          if (r + 8 >= n_valid) { sc[2] = -INFINITY; sc[3] = -INFINITY; }
        }
        if (T > 1 && pos_w + 16 > L - T + 1) {
          // causal limit of the query tokens (virtual head v = head * T + i sees the positions
          // below L - T + 1 + i): only the sequence's last T - 1 positions are masked
          const int cA = 2 * i4, cB = 2 * i4 + 1;   // this lane's QK columns
          const int vA = hg * GW + (GW <= 4 ? (cA & 3) : cA), vB = hg * GW + (GW <= 4 ? (cB & 3) : cB);
          const int limA = L - T + 1 + vA % T, limB = L - T + 1 + vB % T;
          if (pos_w + r >= limA) sc[0] = -INFINITY;
          if (pos_w + r >= limB) sc[1] = -INFINITY;
          if (pos_w + r + 8 >= limA) sc[2] = -INFINITY;
          if (pos_w + r + 8 >= limB) sc[3] = -INFINITY;
        }

        // ---------------- V scales of this lane's PV tokens (2i, 2i+1, 2i+8, 2i+9)
        const int tk[4] = {2 * i4, 2 * i4 + 1, 2 * i4 + 8, 2 * i4 + 9};
        uint32_t dvw[4][C::NB / 2 > 0 ? C::NB / 2 : 1];
        int ex_lane = 0;   // every scale of this lane's tokens is < 2^ex_lane
        if constexpr (C::VQ) {
          uint32_t mx = 0;
  #pragma unroll
          for (int u = 0; u < 4; ++u) {
            load_scale_words<C::NB>(vsc, t0 + tk[u], dvw[u]);
            if (partial && tk[u] >= n_valid) {
  #pragma unroll
              for (int k = 0; k < C::NB / 2; ++k) dvw[u][k] = 0u;
            }
  #pragma unroll
            for (int k = 0; k < C::NB / 2; ++k) mx = __vmaxu2(mx, dvw[u][k]);
          }
          const uint32_t hmax = max(mx & 0xffffu, mx >> 16);   // scales are >= 0: bits order as values
          const int e = (int)(hmax >> 10);
          ex_lane = hmax ? max(e, 1) - 14 : -127;
        }

        // ---------------- lazy online softmax over the warp's 16 tokens (columns = heads)
        const float lm0 = fmaxf(sc[0], sc[2]), lm1 = fmaxf(sc[1], sc[3]);
        const bool over = (lm0 > m0 + kLazy) || (lm1 > m1 + kLazy) || (ex_lane > E);
        if (__any_sync(0xffffffffu, over)) {
          float mx0 = lm0, mx1 = lm1;
          int ex = ex_lane;
  #pragma unroll
          for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
          }
          ex = max(ex, __shfl_xor_sync(0xffffffffu, ex, 1));
          ex = max(ex, __shfl_xor_sync(0xffffffffu, ex, 2));
          const int E_new = max(E, ex);
          const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
          const float e2 = __uint_as_float((uint32_t)(127 + E - E_new) << 23);  // 2^(E - E_new)
          float f0 = (mn0 == -INFINITY) ? 1.0f : fast_exp2(m0 - mn0);
          float f1 = (mn1 == -INFINITY) ? 1.0f : fast_exp2(m1 - mn1);
          l0 *= f0;
          l1 *= f1;
          f0 *= e2;
          f1 *= e2;
  #pragma unroll
          for (int mt = 0; mt < C::QSTEPS; ++mt)
  #pragma unroll
            for (int n = 0; n < C::NPV; ++n) {
              o[mt][n][0] *= f0; o[mt][n][1] *= f1; o[mt][n][2] *= f0; o[mt][n][3] *= f1;
            }
          m0 = mn0;
          m1 = mn1;
          E = E_new;
        }
        // m0, m1 are finite here unless a causal limit masked a column everywhere so far: the
        // warp has a valid token, whose score raised them
        float p0 = fast_exp2(sc[0] - m0);
        float p1 = fast_exp2(sc[1] - m1);
        float p2 = fast_exp2(sc[2] - m0);
        float p3 = fast_exp2(sc[3] - m1);
        if (T > 1) {
          if (sc[0] == -INFINITY) p0 = 0.0f;
          if (sc[1] == -INFINITY) p1 = 0.0f;
          if (sc[2] == -INFINITY) p2 = 0.0f;
          if (sc[3] == -INFINITY) p3 = 0.0f;
        }
        l0 += p0 + p2;
        l1 += p1 + p3;

        // ---------------- transpose p (fp32, as two 16-bit halves) to the PV B layout:
        // lane (r, i) receives p[tok 2i, 2i+1, 2i+8, 2i+9][column r]
        float pv[4];
        {
          const uint32_t u0 = __float_as_uint(p0), u1 = __float_as_uint(p1);
          const uint32_t u2 = __float_as_uint(p2), u3 = __float_as_uint(p3);
          const uint32_t ah = movtrans(__byte_perm(u0, u1, 0x7632)), al = movtrans(__byte_perm(u0, u1, 0x5410));
          const uint32_t bh = movtrans(__byte_perm(u2, u3, 0x7632)), bl = movtrans(__byte_perm(u2, u3, 0x5410));
          pv[0] = __uint_as_float(__byte_perm(al, ah, 0x5410));
          pv[1] = __uint_as_float(__byte_perm(al, ah, 0x7632));
          pv[2] = __uint_as_float(__byte_perm(bl, bh, 0x5410));
          pv[3] = __uint_as_float(__byte_perm(bl, bh, 0x7632));
        }

        // ---------------- PV
        const float pscale = __uint_as_float((uint32_t)(127 + kPScale - E) << 23);  // 2^(kPScale - E)
  #pragma unroll
        for (int u = 0; u < 4; ++u) pv[u] *= pscale;
        // PV column r of an 8-column tile is head r&3's hi part (r < 4) or lo part (r >= 4)
        // when one n-tile carries both; lo lanes feed x - f16(x) instead of x.
        const unsigned short lo_sel = (C::NPV == 1 && r >= 4) ? (C::VBF ? 0xBF80 : 0xBC00) : 0;
        if constexpr (C::VQ) {
          uint32_t vq4[4];   // q4s: one ldmatrix.x4 covers blocks bb and bb + 1 (bb even)
  #pragma unroll
          for (int bb = 0; bb < C::NB; ++bb) {
            float x[4];
  #pragma unroll
            for (int u = 0; u < 4; ++u) {
              const __half hv = __ushort_as_half((unsigned short)(dvw[u][bb >> 1] >> (16 * (bb & 1))));
              x[u] = pv[u] * __half2float(hv);
            }
            uint32_t bf[C::NPV][2];
            if constexpr (C::NPV == 1) {
              bf[0][0] = hi_or_lo<C::VBF>(x[0], x[1], lo_sel);
              bf[0][1] = hi_or_lo<C::VBF>(x[2], x[3], lo_sel);
            } else {
              split2<C::VBF>(x[0], x[1], bf[0][0], bf[1][0]);
              split2<C::VBF>(x[2], x[3], bf[0][1], bf[1][1]);
            }
            if constexpr (VC == KVQ_CODEC_Q8_0) {
              uint32_t y0, y1, y2, y3;
              // matrices: (tok 0-7, chunk 2b), (tok 0-7, chunk 2b+1), (tok 8-15, 2b), (tok 8-15, 2b+1)
              ldsm_x4_t(row_chunk<C::VRB>(vst, t0 + (mi >> 1) * 8 + mr, 2 * bb + (mi & 1)), y0, y1, y2, y3);
              y0 ^= 0x80808080u; y1 ^= 0x80808080u; y2 ^= 0x80808080u; y3 ^= 0x80808080u;
              uint32_t ae[4] = {i8pair_raw(y0, 0x4240), i8pair_raw(y1, 0x4240), i8pair_raw(y2, 0x4240),
                                i8pair_raw(y3, 0x4240)};
              uint32_t ao[4] = {i8pair_raw(y0, 0x4341), i8pair_raw(y1, 0x4341), i8pair_raw(y2, 0x4341),
                                i8pair_raw(y3, 0x4341)};
              // exact small integers in f16 before the product: an offset folded into the fp32
              // accumulator instead loses its low bits there, and that error grows with the chunk
  #pragma unroll
              for (int k = 0; k < 4; ++k) {
                ae[k] = hsub2_u32(ae[k], 0x64806480u);
                ao[k] = hsub2_u32(ao[k], 0x64806480u);
              }
  #pragma unroll
              for (int n = 0; n < C::NPV; ++n) {
                mma16816<false>(o[2 * bb][n], ae, bf[n][0], bf[n][1]);
                mma16816<false>(o[2 * bb + 1][n], ao, bf[n][0], bf[n][1]);
              }
            } else {  // q4s: matrices (tok 0-7, chunk b), (tok 8-15, chunk b) for this block
              if ((bb & 1) == 0)
                ldsm_x4_t(row_chunk<C::VRB>(vst, t0 + (mi & 1) * 8 + mr, bb + (mi >> 1)), vq4[0], vq4[1], vq4[2], vq4[3]);
              const uint32_t ya = (bb & 1) ? vq4[2] : vq4[0], yb = (bb & 1) ? vq4[3] : vq4[1];
              const uint32_t ya8 = ya >> 8, yb8 = yb >> 8;
              // even nibbles: 1024 + u, less 1032; odd nibbles in place: (1024 + 16 u) / 16 - 72
              const uint32_t a01[4] = {hsub2_u32(u4pair_raw(ya), 0x64086408u),
                                       hfma2_u32(u4pair_hi_raw(ya), kSixteenth2, kMinus72x2),
                                       hsub2_u32(u4pair_raw(yb), 0x64086408u),
                                       hfma2_u32(u4pair_hi_raw(yb), kSixteenth2, kMinus72x2)};
              const uint32_t a23[4] = {hsub2_u32(u4pair_raw(ya8), 0x64086408u),
                                       hfma2_u32(u4pair_hi_raw(ya8), kSixteenth2, kMinus72x2),
                                       hsub2_u32(u4pair_raw(yb8), 0x64086408u),
                                       hfma2_u32(u4pair_hi_raw(yb8), kSixteenth2, kMinus72x2)};
  #pragma unroll
              for (int n = 0; n < C::NPV; ++n) {
                mma16816<false>(o[2 * bb][n], a01, bf[n][0], bf[n][1]);
                mma16816<false>(o[2 * bb + 1][n], a23, bf[n][0], bf[n][1]);
              }
            }
          }
        } else {
          // 16-bit V: one B operand for every M-tile; zero the A lanes of tokens past the end
          uint32_t bf[C::NPV][2];
          if constexpr (C::NPV == 1) {
            bf[0][0] = hi_or_lo<C::VBF>(pv[0], pv[1], lo_sel);
            bf[0][1] = hi_or_lo<C::VBF>(pv[2], pv[3], lo_sel);
          } else {
            split2<C::VBF>(pv[0], pv[1], bf[0][0], bf[1][0]);
            split2<C::VBF>(pv[2], pv[3], bf[0][1], bf[1][1]);
          }
          uint32_t kmask_lo = 0xffffffffu, kmask_hi = 0xffffffffu;
          if (partial) {
            kmask_lo = (tk[0] < n_valid ? 0x0000ffffu : 0u) | (tk[1] < n_valid ? 0xffff0000u : 0u);
            kmask_hi = (tk[2] < n_valid ? 0x0000ffffu : 0u) | (tk[3] < n_valid ? 0xffff0000u : 0u);
          }
  #pragma unroll
          for (int mt = 0; mt < C::QSTEPS; ++mt) {
            uint32_t af[4];
            // matrices: (tok 0-7, chunk 2mt), (tok 0-7, chunk 2mt+1), (tok 8-15, 2mt), (tok 8-15, 2mt+1)
            ldsm_x4_t(row_chunk<C::VRB>(vst, t0 + (mi >> 1) * 8 + mr, 2 * mt + (mi & 1)), af[0], af[1], af[2], af[3]);
            af[0] &= kmask_lo; af[1] &= kmask_lo; af[2] &= kmask_hi; af[3] &= kmask_hi;
  #pragma unroll
            for (int n = 0; n < C::NPV; ++n) mma16816<C::VBF>(o[mt][n], af, bf[n][0], bf[n][1]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      if (pw == 0 && tile + C::NS < n_tiles) {
        // refill the stage once every warp has released it; lane 0 issues the copies
        if (!mbar_wait_warp(bar_empty + 8 * s, (tile / C::NS) & 1, wlim)) {
          timed_out = true;
          break;
        }
        const int page = page_of(tile + C::NS);
        if (lane == 0) issue_tile(tile + C::NS, page);
        __syncwarp();
      }
    }
  }
  // ------------------------------------------------------------ merge the warps
  const int NWT = C::NW * 32;
  if (timed_out) {
    record_fault(a.k.status, KVQ_DEVICE_TIMEOUT);
    // Leave no bulk copy in flight into this CTA's shared memory: wait for the phase of the
    // last tile issued into each stage of the pipeline (copies that were issued complete).
    // A stage never issued has nothing in flight and is not waited on.  Every warp that
    // issues a copy records it before its own drain, so each copy is drained by its issuer
    // at least.
    for (int st = 0; st < C::NS; ++st) {
      const int t = last_issued[st];
      if (t >= 0) (void)mbar_wait_warp(bar_full + 8 * st, (t / C::NS) & 1);
    }
  }
  // per-head sums of the lanes' partials; O true scale: O * 2^(E - kPScale)
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, off);
    l1 += __shfl_xor_sync(0xffffffffu, l1, off);
  }
  const float oscale = __uint_as_float((uint32_t)(127 + E - kPScale) << 23);
  const long long head0 = (long long)b * a.num_q_heads + (long long)kvh * G;
  const int gcount = G < GW * HG ? G : GW * HG;
  if (C::LEAN && a.warp_records > 0) {
    // ---- record mode: this warp's partial, in register order (one float2 per lane and
    // M-tile: lanes i < 2 rows r, lanes i >= 2 rows r + 8 after adding the lo columns),
    // and its (m, l) per head; the record merge kernel combines the records
    const long long rec = ((long long)b * gridDim.y + kvh) * a.warp_records + (long long)chunk * C::NW + warp;
    if (r == 0 && i4 < 2) reinterpret_cast<float4*>(a.part_ml + rec * 8)[i4] = make_float4(m0, l0, m1, l1);
    float2* ro = reinterpret_cast<float2*>(a.part_o + rec * (C::QSTEPS * 64)) + lane;
#pragma unroll
    for (int mt = 0; mt < C::QSTEPS; ++mt) {
      float v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = o[mt][0][k] + __shfl_xor_sync(0xffffffffu, o[mt][0][k], 2);
      ro[mt * 32] = i4 < 2 ? make_float2(v[0] * oscale, v[1] * oscale) : make_float2(v[2] * oscale, v[3] * oscale);
    }
    return;
  }
  if constexpr (C::NPV == 1 && HG == 1 && C::NW <= 16) {
    // ---- warps of at most 4 heads: every warp's accumulators have the same lane layout
    // (lane (r, i) holds rows r, r + 8 of each M-tile for columns 2i, 2i + 1, i.e. heads
    // 2(i & 1), 2(i & 1) + 1, hi parts for i < 2 and lo parts for i >= 2), so the warps
    // are summed position by position: each warp stores its scaled values in register
    // order (one float2 per lane and M-tile, no bank conflicts) and thread t adds up
    // position t of every warp.
    float* hml = ml_all + C::NW * 16;        // per-head (M, l) of the whole CTA [4][2]
    float* obuf = reinterpret_cast<float*>(smem);
    if (r == 0) *reinterpret_cast<float4*>(ml_all + warp * 16 + i4 * 4) = make_float4(m0, l0, m1, l1);
    // every warp reaches this barrier (a timed-out warp skips only its tiles); after it
    // all loops are done, so the rings are idle
    asm volatile("bar.sync 1, %0;" ::"r"(NWT) : "memory");
    // (M, l) of heads 2hp, 2hp + 1 over the CTA's warps: lane (hp, w) reads warp w's pair
    const int hp = lane >> 4, wr = lane & 15;
    const float4 mlw = wr < C::NW ? *reinterpret_cast<const float4*>(ml_all + wr * 16 + hp * 4)
                                  : make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
    float Ma = mlw.x, Mb = mlw.z;
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) {
      Ma = fmaxf(Ma, __shfl_xor_sync(0xffffffffu, Ma, off));
      Mb = fmaxf(Mb, __shfl_xor_sync(0xffffffffu, Mb, off));
    }
    float la = mlw.x == -INFINITY ? 0.0f : fast_exp2(mlw.x - Ma) * mlw.y;
    float lb = mlw.z == -INFINITY ? 0.0f : fast_exp2(mlw.z - Mb) * mlw.w;
#pragma unroll
    for (int off = 1; off < 16; off <<= 1) {
      la += __shfl_xor_sync(0xffffffffu, la, off);
      lb += __shfl_xor_sync(0xffffffffu, lb, off);
    }
    if (warp == 0 && wr == 0) *reinterpret_cast<float4*>(hml + hp * 4) = make_float4(Ma, la, Mb, lb);
    {
      const int src = (i4 & 1) * 16;          // the lane holding this lane's head pair
      const float MA = __shfl_sync(0xffffffffu, Ma, src), MB = __shfl_sync(0xffffffffu, Mb, src);
      const float mA = __shfl_sync(0xffffffffu, m0, (lane & ~3) | (i4 & 1));
      const float mB = __shfl_sync(0xffffffffu, m1, (lane & ~3) | (i4 & 1));
      const float fA = (mA == -INFINITY) ? 0.0f : fast_exp2(mA - MA) * oscale;
      const float fB = (mB == -INFINITY) ? 0.0f : fast_exp2(mB - MB) * oscale;
#pragma unroll
      for (int mt = 0; mt < C::QSTEPS; ++mt) {
        float v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) v[k] = o[mt][0][k] + __shfl_xor_sync(0xffffffffu, o[mt][0][k], 2);
        // lanes i < 2 keep rows r (d0), lanes i >= 2 rows r + 8 (d1)
        const float2 w2 = i4 < 2 ? make_float2(v[0] * fA, v[1] * fB) : make_float2(v[2] * fA, v[3] * fB);
        *reinterpret_cast<float2*>(obuf + (warp * C::QSTEPS + mt) * 64 + lane * 2) = w2;
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NWT) : "memory");
    // position t = (M-tile, lane, k) -> (head, element of head_dim)
    for (int t = tid; t < C::QSTEPS * 64; t += NWT) {
      const int mt = t >> 6, ln = (t >> 1) & 31, k = t & 1;
      const int rr = ln >> 2, ii = ln & 3;
      const int dim = pv_dim<VC>(mt, ii < 2 ? rr : rr + 8);
      const int h = 2 * (ii & 1) + k;
      if (h >= gcount) continue;
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < C::NW; ++w) sum += obuf[(w * C::QSTEPS + mt) * 64 + (t & 63)];
      if (nv == 1) {
        // the whole sequence is this chunk: normalize and write the output (no split)
        const float lsum = hml[2 * h + 1];
        a.out[(head0 + h) * D + dim] = lsum > 0.0f ? sum / lsum : 0.0f;
      } else {
        a.part_o[((head0 + h) * a.n_chunks + chunk) * D + dim] = sum;   // partial write (a7)
      }
    }
    if (nv == 1) {
      return;
    }
    if (tid < gcount) {
      a.part_ml[((head0 + tid) * a.n_chunks + chunk) * 2] = hml[2 * tid];
      a.part_ml[((head0 + tid) * a.n_chunks + chunk) * 2 + 1] = hml[2 * tid + 1];
    }
  } else {
    float* ml = ml_all + warp * 16;   // its own region (not part of the rings)
    if (r == 0) {
      ml[(2 * i4) * 2] = m0;
      ml[(2 * i4) * 2 + 1] = l0;
      ml[(2 * i4 + 1) * 2] = m1;
      ml[(2 * i4 + 1) * 2 + 1] = l1;
    }
    // every warp reaches this barrier (a timed-out warp skips only its tiles); after it all
    // loops are done, so the rings are idle
    asm volatile("bar.sync 1, %0;" ::"r"(NWT) : "memory");
    float* obuf = reinterpret_cast<float*>(smem);
    // warp index of member w of head group hgi in pipeline pp
    auto wix = [&](int pp, int hgi, int w) { return pp * C::PW + hgi * 4 + w; };
    float* hml = ml_all + C::NW * 16;     // per-head (M, l) of the whole CTA [16][2]
    if (warp == 0 && lane < gcount) {
      const int h = lane, hgi = h / GW, hl = h % GW;
      float M = -INFINITY;
      for (int pp = 0; pp < C::NP; ++pp)
        for (int w = 0; w < 4; ++w) M = fmaxf(M, ml_all[wix(pp, hgi, w) * 16 + hl * 2]);
      float lsum = 0.0f;
      for (int pp = 0; pp < C::NP; ++pp)
        for (int w = 0; w < 4; ++w) {
          const float mw = ml_all[wix(pp, hgi, w) * 16 + hl * 2];
          if (mw != -INFINITY) lsum += fast_exp2(mw - M) * ml_all[wix(pp, hgi, w) * 16 + hl * 2 + 1];
        }
      hml[2 * h] = M;
      hml[2 * h + 1] = lsum;
    }
    {
      // heads of this lane's O columns after folding: 2*i4, 2*i4+1 (lanes i4 < GW/2 only)
      const int hA = 2 * i4, hB = 2 * i4 + 1;
      float fA = 0.0f, fB = 0.0f;
      {
        // over the warps of this head group in every pipeline
        float MA = -INFINITY, MB = -INFINITY;
  #pragma unroll
        for (int pp = 0; pp < C::NP; ++pp)
  #pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int wi = wix(pp, hg, w);
            MA = fmaxf(MA, ml_all[wi * 16 + (hA & 7) * 2]);
            MB = fmaxf(MB, ml_all[wi * 16 + (hB & 7) * 2]);
          }
        const float mA = __shfl_sync(0xffffffffu, m0, (lane & ~3) | (i4 & (GW <= 4 ? 1 : 3)));
        const float mB = __shfl_sync(0xffffffffu, m1, (lane & ~3) | (i4 & (GW <= 4 ? 1 : 3)));
        fA = (mA == -INFINITY) ? 0.0f : fast_exp2(mA - MA) * oscale;
        fB = (mB == -INFINITY) ? 0.0f : fast_exp2(mB - MB) * oscale;
      }
  #pragma unroll
      for (int mt = 0; mt < C::QSTEPS; ++mt) {
        float v[4];
  #pragma unroll
        for (int k = 0; k < 4; ++k) {
          float x = o[mt][0][k];
          if constexpr (C::NPV == 2) x += o[mt][1][k];
          else x += __shfl_xor_sync(0xffffffffu, x, 2);  // add the lo columns (lanes i4 ^ 2)
          v[k] = x;
        }
        if (GW > 4 || i4 < 2) {
          const int d0 = pv_dim<VC>(mt, r), d1 = pv_dim<VC>(mt, r + 8);
          obuf[(warp * 8 + hA) * D + d0] = v[0] * fA;
          obuf[(warp * 8 + hB) * D + d0] = v[1] * fB;
          obuf[(warp * 8 + hA) * D + d1] = v[2] * fA;
          obuf[(warp * 8 + hB) * D + d1] = v[3] * fB;
        }
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(NWT) : "memory");
    if (nv == 1) {
      // the whole sequence is this chunk: normalize and write the output (no split)
      for (int idx = tid; idx < gcount * D; idx += NWT) {
        const int h = idx / D, j = idx % D;
        const int hgi = h / GW, hl = h % GW;
        float sum = 0.0f;
  #pragma unroll
        for (int pp = 0; pp < C::NP; ++pp)
  #pragma unroll
          for (int w = 0; w < 4; ++w) sum += obuf[(wix(pp, hgi, w) * 8 + hl) * D + j];
        const float lsum = hml[2 * h + 1];
        a.out[(head0 + h) * D + j] = lsum > 0.0f ? sum / lsum : 0.0f;
      }
      return;
    }
    // ------------------------------------------------------------ partial write (a7)
    for (int idx = tid; idx < gcount * D; idx += NWT) {
      const int h = idx / D, j = idx % D;
      const int hgi = h / GW, hl = h % GW;
      float sum = 0.0f;
  #pragma unroll
      for (int pp = 0; pp < C::NP; ++pp)
  #pragma unroll
        for (int w = 0; w < 4; ++w) sum += obuf[(wix(pp, hgi, w) * 8 + hl) * D + j];
      a.part_o[((head0 + h) * a.n_chunks + chunk) * D + j] = sum;
    }
    for (int h = tid; h < gcount; h += NWT) {
      a.part_ml[((head0 + h) * a.n_chunks + chunk) * 2] = hml[2 * h];
      a.part_ml[((head0 + h) * a.n_chunks + chunk) * 2 + 1] = hml[2 * h + 1];
    }
  }
  // ------------------------------------------------------------ split-K combine (a8)
  split_k_combine<D, C::NW>(a, smem, reinterpret_cast<volatile int*>(smem + C::OK_OFF) + 16, b, kvh, chunk, nv,
                            head0, gcount);
  }   // tokens-on-M loop
}

template <int KC, int VC, int D, int GW, int HG, bool SOLO>
__global__ void __launch_bounds__(Cfg<KC, VC, D, GW, HG, SOLO>::THREADS, Cfg<KC, VC, D, GW, HG, SOLO>::MINB)
decode_mma_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  DecodeArgs a) {
  decode_cta<KC, VC, D, GW, HG, SOLO>(tmk, tmv, a);
}

// Sets the kernel's shared-memory attributes once per device.
template <int KC, int VC, int D, int GW, int HG, bool SOLO>
cudaError_t prepare() {
  using C = Cfg<KC, VC, D, GW, HG, SOLO>;
  static unsigned long long done = 0;   // bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && (done >> dev) & 1ull) return cudaSuccess;
  auto kern = decode_mma_kernel<KC, VC, D, GW, HG, SOLO>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_RELAXED);
  return e;
}

template <int KC, int VC, int D, int GW, int HG, bool SOLO = false>
cudaError_t launch(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream) {
  using C = Cfg<KC, VC, D, GW, HG, SOLO>;
  auto kern = decode_mma_kernel<KC, VC, D, GW, HG, SOLO>;
  cudaError_t e = prepare<KC, VC, D, GW, HG, SOLO>();
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_chunks, a.k.num_kv_heads, a.batch);
  e = launch_pdl(kern, grid, dim3(C::THREADS), C::SMEM, stream, tmk, tmv, a);
  count_launch();
  return e;
}

// Resident CTAs per SM of one instantiation (0 on error); *pipes = its pipelines per CTA.
template <int KC, int VC, int D, int GW, int HG, bool SOLO = false>
int occupancy(int* pipes) {
  using C = Cfg<KC, VC, D, GW, HG, SOLO>;
  auto kern = decode_mma_kernel<KC, VC, D, GW, HG, SOLO>;
  *pipes = C::NP;
  if (prepare<KC, VC, D, GW, HG, SOLO>() != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, C::SMEM) != cudaSuccess) return 0;
  return n;
}

// The heads-on-M loop serves 9..32 query rows per KV head for q8_0 K and V at head_dim
// 128 and 256; other shapes take the tokens-on-M loop (up to 16 rows).
template <int KC, int VC>
constexpr bool kHeadsOnM = KC == KVQ_CODEC_Q8_0 && VC == KVQ_CODEC_Q8_0;

template <int KC, int VC>
int occupancy_pair(int head_dim, int g, int* pipes, bool solo) {
#define KVQ_MMA_O(D)                                                               \
  if constexpr (D <= 128) {                                                        \
    if (g <= 4 && solo) return occupancy<KC, VC, D, 4, 1, true>(pipes);            \
  }                                                                                \
  if (g <= 4) return occupancy<KC, VC, D, 4, 1>(pipes);                            \
  if (g <= 8) return occupancy<KC, VC, D, 8, 1>(pipes);                            \
  if constexpr (kHeadsOnM<KC, VC> && D >= 128) {                                   \
    if (g <= 16) return occupancy<KC, VC, D, 16, 1>(pipes);                        \
    if (g <= 32) return occupancy<KC, VC, D, 16, 2>(pipes);                        \
  } else {                                                                         \
    if (g <= 16) return occupancy<KC, VC, D, 8, 2>(pipes);                         \
  }                                                                                \
  return 0;
  switch (head_dim) {
    case 64: { KVQ_MMA_O(64) }
    case 128: { KVQ_MMA_O(128) }
    case 256: { KVQ_MMA_O(256) }
    default: return 0;
  }
#undef KVQ_MMA_O
}

template <int KC, int VC>
cudaError_t launch_pair(const DecodeArgs& a, int head_dim, const CUtensorMap& tmk, const CUtensorMap& tmv,
                        cudaStream_t stream) {
  const int g = a.group;
#define KVQ_MMA_G(D)                                                               \
  if constexpr (D <= 128) {                                                        \
    if (g <= 4 && a.solo) return launch<KC, VC, D, 4, 1, true>(a, tmk, tmv, stream); \
  }                                                                                \
  if (g <= 4) return launch<KC, VC, D, 4, 1>(a, tmk, tmv, stream);                \
  if (g <= 8) return launch<KC, VC, D, 8, 1>(a, tmk, tmv, stream);                \
  if constexpr (kHeadsOnM<KC, VC> && D >= 128) {                                   \
    if (g <= 16) return launch<KC, VC, D, 16, 1>(a, tmk, tmv, stream);             \
    if (g <= 32) return launch<KC, VC, D, 16, 2>(a, tmk, tmv, stream);             \
  } else {                                                                         \
    if (g <= 16) return launch<KC, VC, D, 8, 2>(a, tmk, tmv, stream);              \
  }                                                                                \
  return cudaErrorNotSupported;
  switch (head_dim) {
    case 64: { KVQ_MMA_G(64) }
    case 128: { KVQ_MMA_G(128) }
    case 256: { KVQ_MMA_G(256) }
    default: return cudaErrorNotSupported;
  }
#undef KVQ_MMA_G
}

}  // namespace mma
}  // namespace kvq
