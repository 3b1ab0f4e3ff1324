// Chunked prefill attention on the 5th-generation tensor cores (tcgen05, operands and
// accumulators in tensor memory), head_dim 128, K and V each q8_0, q4s or f16, or bf16 /
// bf16, q8_0 / bf16 and q4s / bf16 (a bf16 side takes bf16 operands: Q for a bf16 K, P for
// a bf16 V): the prompt-processing arm of halobench record clm-0022's depth tables (pp512 at
// depth), with the dequantization fused into the load of each KV tile.
//
// A CTA owns 128 query rows of one (sequence, KV head), row = token * G + head-in-group,
// one per tensor-memory lane.  Per 64-token KV tile:
//  * the tile arrives by TMA in the swizzled layout that the MMA reads (16-bit codecs); a
//    q8_0 or q4s tile is turned, once for all 128 rows, into two f16 tiles of that layout
//    that give d q exactly (hi = d q rounded, lo = its rounding error, exact in f16: d has
//    11 significant bits and q at most 7; lo is stored negated and read with the MMA's
//    negate-B bit), with a power of two 2^-sigma folded in per tile (from the tile's largest
//    scale) that keeps every hi below 2^15;
//  * S = Q K^T: M 128 x N 64 x K 128, Q in tensor memory, two MMAs per K step for a quantized
//    K (hi and lo), into one of two 64-column score buffers;
//  * softmax by row (two threads per row, one per 32-score half, the row maximum traded
//    through shared memory under an mbarrier of the warp pair; base 2, lazy running maximum
//    as in the decode kernels); P goes to tensor memory as 16-bit hi + lo (P = P_h + P_l to
//    ~22 bits in f16, ~16 in bf16);
//  * O += P V: M 128 x N 128 x K 64, V as an MN-major operand straight from the tile layout;
//    P_h V_h + P_l V_h (+ P_h V_l for a quantized V), O in 128 tensor-memory columns.  A
//    quantized V tile carries its own 2^-sigma; O is kept in units of the largest sigma so
//    far and rescaled (with the lazy maximum's rescale) when it grows.
// Warp roles, linked by mbarriers only (no CTA-wide barrier inside the tile loop):
//  warps 0-7 softmax (warp w: rows 32 (w % 4) .. + 31, its tensor-memory lanes, score half
//  w / 4), warp 8 issues the MMAs (S of tile t, then PV of tile t - 1, so the tensor cores
//  compute S(t) during the softmax of tile t - 1), warp 9 loads tiles, warps 10-17 convert
//  q8_0 / q4s tiles (double buffered).  Every wait is bounded; a wait that runs out raises a
//  CTA-wide abort flag that the other waits watch, and the timeout is reported in the K
//  store's status word.
#pragma once

#include "kvq_decode_mma.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace prefill_tc {

using namespace kvq::mma;

constexpr int kD = 128;
constexpr int kRows = 128;              // query rows per CTA = tensor-memory lanes
constexpr int kTile16 = kT * kD * 2;    // one 64 x 128 f16 operand tile (16 KB)
constexpr int kTmemCols = 512;
// tensor-memory columns: S buffers 0 and 64, O 128, P buffers (hi 32, lo 32) 256 and 320, Q 384
constexpr uint32_t kColO = 128, kColP = 256, kColQ = 384;
constexpr int kSoftmaxWarps = 8, kMmaWarp = 8, kLoadWarp = 9, kConvWarp0 = 10, kConvWarps = 8;

template <int KC, int VC>
struct TCfg {
  static constexpr bool K4 = KC == KVQ_CODEC_Q4S, V4 = VC == KVQ_CODEC_Q4S;   // 4-bit codes
  static constexpr bool KQ = KC == KVQ_CODEC_Q8_0 || K4, VQ = VC == KVQ_CODEC_Q8_0 || V4, CONV = KQ || VQ;
  // 16-bit types of the two products: bf16 when that side's 16-bit operand is bf16 (Q and
  // a bf16 K; P and a bf16 V), f16 otherwise
  static constexpr bool SBF = KC == KVQ_CODEC_BF16, PBF = VC == KVQ_CODEC_BF16;
  static constexpr int THREADS = 32 * (CONV ? kConvWarp0 + kConvWarps : kConvWarp0);
  static constexpr int NB = kD / kBlock;
  static constexpr int KRB = K4 ? kD / 2 : KQ ? kD : 2 * kD, VRB = V4 ? kD / 2 : VQ ? kD : 2 * kD;
  static constexpr int KROWS = kT * KRB, VROWS = kT * VRB;
  static constexpr int KSC = KQ ? kT * NB * 2 : 0, VSC = VQ ? kT * NB * 2 : 0;
  static constexpr int V_OFF = KROWS, KSC_OFF = KROWS + VROWS, VSC_OFF = KSC_OFF + KSC;
  static constexpr int al1k(int x) { return (x + 1023) / 1024 * 1024; }
  static constexpr int STAGE = al1k(KROWS + VROWS + KSC + VSC);
  static constexpr int FIXED = (KQ ? 4 * kTile16 : 0) + (VQ ? 4 * kTile16 : 0) + 2048 + 3 * 2 * kRows * 4;
  static constexpr int NST0 = (227 * 1024 - 1024 - FIXED) / STAGE;
  static constexpr int NST = NST0 > 6 ? 6 : NST0;                 // TMA stages
  static constexpr int KC_OFF = NST * STAGE;                       // converted K: 2 x (hi, lo)
  static constexpr int VC_OFF = KC_OFF + (KQ ? 4 * kTile16 : 0);   // converted V: 2 x (hi, lo)
  static constexpr int BAR_OFF = VC_OFF + (VQ ? 4 * kTile16 : 0);
  // barriers: full[NST], empty[NST], then pairs kc_full, kc_empty, vc_full, vc_empty, s_full,
  // s_empty, p_full, p_empty, then q_full, drain, then the softmax row pairs' exchanges
  // (per pair of warps: two tile parities and the final sums)
  static constexpr int NBAR = 2 * NST + 16 + 2 + 12;
  static constexpr int MISC_OFF = BAR_OFF + 8 * NBAR;              // tensor-memory base, abort, stage flags
  static constexpr int RED_OFF = MISC_OFF + 64;                    // row maxima [2 tiles][2 halves][rows], sums
  static constexpr int SMEM = RED_OFF + 3 * 2 * kRows * 4 + 1024;
  static constexpr uint32_t TX = KROWS + VROWS + KSC + VSC;
  // arrivals that release a stage: softmax warps (flags, scales), converter warps, and the
  // MMA warp's commit when an MMA reads the stage itself
  static constexpr int EMPTY_COUNT = kSoftmaxWarps + (CONV ? kConvWarps : 0) + (KQ && VQ ? 0 : 1);
  static_assert(NST >= 3 && SMEM <= 227 * 1024, "shared memory");
};

// Byte offset of 16-byte chunk `c` (8 elements of 16 bits) of row `t` in a tile of 64-row
// regions of 128-byte lines (the TMA layout): region c / 8.
__device__ __forceinline__ uint32_t tile_chunk(int t, int c) {
  return (uint32_t)((c >> 3) * (kT * 128) + t * 128 + (((c & 7) ^ (t & 7)) << 4));
}

// Per-tile prescale exponent of a q8_0 tile: sigma = e - 22 for the largest scale's biased
// f16 exponent e over the valid rows, so d 2^-sigma < 2^8 and |d q| 2^-sigma < 2^15.
// Every warp forms the same value from the same 512 bytes of scales.
__device__ __forceinline__ int tile_sigma(const uint8_t* sc, int lane, int n_valid) {
  const uint4 w = *reinterpret_cast<const uint4*>(sc + lane * 16);   // rows 2 lane, 2 lane + 1
  uint32_t m0 = max(max(w.x & 0x7FFFu, w.x >> 16 & 0x7FFFu), max(w.y & 0x7FFFu, w.y >> 16 & 0x7FFFu));
  uint32_t m1 = max(max(w.z & 0x7FFFu, w.z >> 16 & 0x7FFFu), max(w.w & 0x7FFFu, w.w >> 16 & 0x7FFFu));
  if (2 * lane >= n_valid) m0 = 0u;
  if (2 * lane + 1 >= n_valid) m1 = 0u;
  const uint32_t m = __reduce_max_sync(0xffffffffu, max(m0, m1));
  return (int)(m >> 10) - 22;
}

// Shared-memory offsets of one 16-code chunk a converter thread handles in every tile: the
// codes (TMA layout), its scale, and its two 16-byte destinations (the two-region layout).
struct ConvItem {
  uint32_t src, scale, dst0, dst1;
  int row;
};
__device__ __forceinline__ ConvItem conv_item(int i) {
  const int t = i >> 3, c = i & 7;   // row, 16-code chunk
  return {(uint32_t)(t * 128 + ((c ^ (t & 7)) << 4)), (uint32_t)((t * 4 + (c >> 1)) * 2), tile_chunk(t, 2 * c),
          tile_chunk(t, 2 * c + 1), t};
}

// q8_0 tile (TMA layout, one 128-byte line per row) + its scales -> f16 hi and negated lo
// tiles of the two-region layout, d q 2^-sigma = hi - nlo exactly (nlo = hi - d q 2^-sigma,
// the product's rounding error with its sign flipped: the MMAs that read it negate B);
// rows >= n_valid become zeros.
template <int NI>
__device__ __forceinline__ void convert_q8(const uint8_t* rows, const uint8_t* sc, uint8_t* dst, const ConvItem* it,
                                           int n_valid, int sigma) {
  const float f = __uint_as_float((uint32_t)(127 - sigma) << 23);
#pragma unroll
  for (int u = 0; u < NI; ++u) {
    uint32_t hi[8], lo[8];
    if (it[u].row < n_valid) {
      const uint4 w = *reinterpret_cast<const uint4*>(rows + it[u].src);
      const float d = __half2float(*reinterpret_cast<const __half*>(sc + it[u].scale)) * f;
      const uint32_t d2 = pack2<false>(d, d), nd2 = d2 ^ 0x80008000u;
      const uint32_t ws[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t q2 = hsub2_u32(i8pair_raw(ws[k >> 1], (k & 1) ? 0x4342 : 0x4140), 0x64806480u);
        __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&q2), *reinterpret_cast<const __half2*>(&d2));
        hi[k] = *reinterpret_cast<uint32_t*>(&h);
        lo[k] = hfma2_u32(q2, nd2, hi[k]);   // hi - d q, exact
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) hi[k] = lo[k] = 0u;
    }
    *reinterpret_cast<uint4*>(dst + it[u].dst0) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(dst + it[u].dst1) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    *reinterpret_cast<uint4*>(dst + kTile16 + it[u].dst0) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(dst + kTile16 + it[u].dst1) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  }
}

// The same for a q4s tile: rows of 64 bytes (TMA's 64-byte swizzle: 16-byte chunk c of row t
// at c ^ ((t >> 1) & 3)), chunk c = block c = dims 32 c .. 32 c + 31, byte j of it holding
// dims 2 j (low nibble) and 2 j + 1 (high nibble) as q + 8.
struct Conv4Item {
  uint32_t src, scale, dst[4];
  int row;
};
__device__ __forceinline__ Conv4Item conv4_item(int i) {
  const int t = i >> 2, c = i & 3;   // row, 32-code block
  Conv4Item it;
  it.src = (uint32_t)(t * 64 + ((c ^ ((t >> 1) & 3)) << 4));
  it.scale = (uint32_t)((t * 4 + c) * 2);
#pragma unroll
  for (int j = 0; j < 4; ++j) it.dst[j] = tile_chunk(t, 4 * c + j);
  it.row = t;
  return it;
}
constexpr uint32_t kQ4Mul = 0x2C003C00u;   // f16 pair (1, 1/16)
constexpr uint32_t kQ4Add = 0xD480E408u;   // f16 pair (-1032, -72)
template <int NI>
__device__ __forceinline__ void convert_q4(const uint8_t* rows, const uint8_t* sc, uint8_t* dst, const Conv4Item* it,
                                           int n_valid, int sigma) {
  const float f = __uint_as_float((uint32_t)(127 - sigma) << 23);
#pragma unroll
  for (int u = 0; u < NI; ++u) {
    uint32_t hi[16], lo[16];
    if (it[u].row < n_valid) {
      const uint4 w = *reinterpret_cast<const uint4*>(rows + it[u].src);
      const float d = __half2float(*reinterpret_cast<const __half*>(sc + it[u].scale)) * f;
      const uint32_t d2 = pack2<false>(d, d), nd2 = d2 ^ 0x80008000u;
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        // byte j twice, as (1024 + low nibble, 1024 + 16 high nibble), then both codes exactly
        const uint32_t y = __byte_perm(ws[j >> 2], 0u, 0x4040u + 0x0101u * (uint32_t)(j & 3));
        const uint32_t q2 = hfma2_u32(and_or(y, 0x00F0000Fu, 0x64006400u), kQ4Mul, kQ4Add);
        __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&q2), *reinterpret_cast<const __half2*>(&d2));
        hi[j] = *reinterpret_cast<uint32_t*>(&h);
        lo[j] = hfma2_u32(q2, nd2, hi[j]);   // hi - d q, exact
      }
    } else {
#pragma unroll
      for (int j = 0; j < 16; ++j) hi[j] = lo[j] = 0u;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      *reinterpret_cast<uint4*>(dst + it[u].dst[j]) = make_uint4(hi[4 * j], hi[4 * j + 1], hi[4 * j + 2], hi[4 * j + 3]);
      *reinterpret_cast<uint4*>(dst + kTile16 + it[u].dst[j]) =
          make_uint4(lo[4 * j], lo[4 * j + 1], lo[4 * j + 2], lo[4 * j + 3]);
    }
  }
}

// Bounded wait of a whole warp for the phase of parity `parity`; gives up (false) at the
// limit, raising the abort flag, or as soon as another role has raised it.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag, int limit) {
  for (int it = 0; it < limit; ++it) {
    if (__all_sync(0xffffffffu, mbar_try(bar, parity))) return true;
    if (*abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}
// One arrival per warp (lane 0, after the warp's own work).
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

template <int KC, int VC>
__global__ void __launch_bounds__(TCfg<KC, VC>::THREADS, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  PrefillArgs a) {
  using C = TCfg<KC, VC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + C::BAR_OFF;
  const uint32_t bar_full = bars, bar_empty = bars + 8 * C::NST;
  const uint32_t pairs = bar_empty + 8 * C::NST;   // each pair: buffer 0, buffer 1
  const uint32_t kc_full = pairs, kc_empty = pairs + 16, vc_full = pairs + 32, vc_empty = pairs + 48;
  const uint32_t s_full = pairs + 64, s_empty = pairs + 80, p_full = pairs + 96, p_empty = pairs + 112;
  const uint32_t q_full = pairs + 128, bar_drain = pairs + 136, xch = pairs + 144;   // xch: [4][3]
  const int wl = a.wait_limit;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 1);
  volatile int* stage_ok = reinterpret_cast<volatile int*>(misc + 4);

  const int rt = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.group, T = a.tokens, P = a.k.page_size;
  const int rows_total = T * G;
  const int row0 = rt * kRows;

  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const int32_t* pt = a.page_table + (long long)b * a.max_pages;
  long long L = a.seq_lens[b];
  const long long cap = (long long)a.max_pages * P;
  if (L < 0 || L > cap) {
    if (tid == 0 && rt == 0 && kvh == 0) {
      record_fault(a.k.status, KVQ_DEVICE_BAD_SEQ_LEN);
      record_fault(a.v.status, KVQ_DEVICE_BAD_SEQ_LEN);
    }
    L = L < 0 ? 0 : cap;
  }
  const int i_last = min(row0 + kRows - 1, rows_total - 1) / G;
  const long long kv_end_ll = min(L, L - T + i_last + 1);
  const int kv_end = kv_end_ll > 0 ? (int)kv_end_ll : 0;
  const int n_tiles = (kv_end + kT - 1) / kT;

  if (tid == 0) {
    for (int s = 0; s < C::NST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, C::EMPTY_COUNT);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(kc_full + 8 * i, kConvWarps);
      mbar_init(kc_empty + 8 * i, 1);
      mbar_init(vc_full + 8 * i, kConvWarps);
      mbar_init(vc_empty + 8 * i, 1);
      mbar_init(s_full + 8 * i, 1);
      mbar_init(s_empty + 8 * i, kSoftmaxWarps);
      mbar_init(p_full + 8 * i, kSoftmaxWarps);
      mbar_init(p_empty + 8 * i, 1);
    }
    mbar_init(q_full, kSoftmaxWarps);
    mbar_init(bar_drain, 1);
    for (int i = 0; i < 12; ++i) mbar_init(xch + 8 * i, 2);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(sbase + C::MISC_OFF, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = misc[0];

  auto nv_of = [&](int t) -> int {   // valid rows of tile t (none when its page was bad)
    return stage_ok[t % C::NST] ? min(kT, kv_end - t * kT) : 0;
  };

  if (warp == kLoadWarp) {
    // ---------------------------------------------------------------- TMA producer
    auto load_page = [&](int tile) -> int {
      const long long pos0 = (long long)tile * kT;
      return pos0 < cap ? __ldg(pt + pos0 / P) : -1;
    };
    int pg_lo = load_page(lane), pg_hi = load_page(32 + lane), pb = 0;
    int issued = 0;
    for (; issued < n_tiles; ++issued) {
      const int t = issued, s = t % C::NST;
      if (t >= C::NST && !wait_phase(bar_empty + 8 * s, ((t / C::NST) - 1) & 1, abort_flag, wl)) break;
      if (t == a.skip_tile) continue;   // fault injection: never issued (no copy, no arrival)
      while (t >= pb + 32) {
        pg_lo = pg_hi;
        pb += 32;
        pg_hi = load_page(pb + 32 + lane);
      }
      const int page = __shfl_sync(0xffffffffu, pg_lo, t - pb);
      if (lane == 0) {
        const int rr0 = (t * kT) % P;
        const uint32_t full = bar_full + 8 * s;
        const bool ok = page >= 0 && page < a.k.num_pages && page < a.v.num_pages;
        stage_ok[s] = ok ? 1 : 0;
        if (!ok) {
          record_fault(a.k.status, KVQ_DEVICE_BAD_PAGE);
          record_fault(a.v.status, KVQ_DEVICE_BAD_PAGE);
          mbar_arrive(full);
        } else {
          mbar_expect_tx(full, C::TX);
          const uint32_t st = sbase + s * C::STAGE;
#pragma unroll
          for (int seg = 0; seg < (C::KRB + 127) / 128; ++seg)
            tma_load_4d(st + seg * kT * 128, &tmk, seg * 128, rr0, kvh, page, full);
#pragma unroll
          for (int seg = 0; seg < (C::VRB + 127) / 128; ++seg)
            tma_load_4d(st + C::V_OFF + seg * kT * 128, &tmv, seg * 128, rr0, kvh, page, full);
          if constexpr (C::KQ)
            bulk_load(st + C::KSC_OFF, a.k.buf + ((long long)page * a.k.num_kv_heads + kvh) * a.k.slab_bytes +
                                           (long long)P * C::KRB + (long long)rr0 * C::NB * 2,
                      kT * C::NB * 2, full);
          if constexpr (C::VQ)
            bulk_load(st + C::VSC_OFF, a.v.buf + ((long long)page * a.v.num_kv_heads + kvh) * a.v.slab_bytes +
                                           (long long)P * C::VRB + (long long)rr0 * C::NB * 2,
                      kT * C::NB * 2, full);
        }
      }
      __syncwarp();
    }
    if (*abort_flag) {
      // copies still in flight land before the CTA leaves (bounded)
      for (int t = max(0, issued - C::NST); t < issued; ++t)
        mbar_wait_warp(bar_full + 8 * (t % C::NST), (t / C::NST) & 1, 1 << 16);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA issue
    const uint32_t idS = tc::idesc_f16(kRows, kT, false, C::SBF), idO = tc::idesc_f16(kRows, kD, true, C::PBF);
    bool ok = wait_phase(q_full, 0, abort_flag, wl);
    tc::fence_after_sync();
    for (int t = 0; ok && t <= n_tiles; ++t) {
      if (t < n_tiles) {   // S(t) into score buffer t & 1
        const int bb = t & 1;
        ok = C::KQ ? wait_phase(kc_full + 8 * bb, (t >> 1) & 1, abort_flag, wl)
                   : wait_phase(bar_full + 8 * (t % C::NST), (t / C::NST) & 1, abort_flag, wl);
        if (ok && t >= 2) ok = wait_phase(s_empty + 8 * bb, ((t >> 1) - 1) & 1, abort_flag, wl);
        if (!ok) break;
        tc::fence_after_sync();
        if (lane == 0) {
          const uint32_t kb = C::KQ ? sbase + C::KC_OFF + bb * 2 * kTile16 : sbase + (t % C::NST) * C::STAGE;
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks) {
            const uint64_t bd = tc::sdesc_sw128(kb + (ks >> 2) * (kT * 128) + (ks & 3) * 32, 16, 1024);
            tc::mma_f16_ta(tmem + 64 * bb, tmem + kColQ + 8 * ks, bd, idS, ks > 0);
            if constexpr (C::KQ) {
              const uint64_t bl = tc::sdesc_sw128(kb + kTile16 + (ks >> 2) * (kT * 128) + (ks & 3) * 32, 16, 1024);
              tc::mma_f16_ta(tmem + 64 * bb, tmem + kColQ + 8 * ks, bl, idS | tc::kNegateB, true);   // negated lo
            }
          }
          tc::mma_commit(s_full + 8 * bb);
          if constexpr (C::KQ) tc::mma_commit(kc_empty + 8 * bb);
        }
        __syncwarp();
      }
      if (t >= 1) {   // PV(t - 1)
        const int u = t - 1, bb = u & 1;
        ok = wait_phase(p_full + 8 * bb, (u >> 1) & 1, abort_flag, wl);
        if (ok) {
          if constexpr (C::VQ) ok = wait_phase(vc_full + 8 * bb, (u >> 1) & 1, abort_flag, wl);
          else ok = wait_phase(bar_full + 8 * (u % C::NST), (u / C::NST) & 1, abort_flag, wl);
        }
        if (!ok) break;
        tc::fence_after_sync();
        if (lane == 0) {
          const uint32_t vb = C::VQ ? sbase + C::VC_OFF + bb * 2 * kTile16 : sbase + (u % C::NST) * C::STAGE + C::V_OFF;
          const uint32_t ph = tmem + kColP + 64 * bb, pl = ph + 32;
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk) {
            const uint64_t bh = tc::sdesc_sw128(vb + kk * 2048, kT * 128, 1024);
            tc::mma_f16_ta(tmem + kColO, ph + 8 * kk, bh, idO, u > 0 || kk > 0);
            tc::mma_f16_ta(tmem + kColO, pl + 8 * kk, bh, idO, true);
            if constexpr (C::VQ) {
              const uint64_t bl = tc::sdesc_sw128(vb + kTile16 + kk * 2048, kT * 128, 1024);
              tc::mma_f16_ta(tmem + kColO, ph + 8 * kk, bl, idO | tc::kNegateB, true);   // negated lo
            }
          }
          tc::mma_commit(p_empty + 8 * bb);
          if constexpr (C::VQ) tc::mma_commit(vc_empty + 8 * bb);
          if constexpr (!(C::KQ && C::VQ)) tc::mma_commit(bar_empty + 8 * (u % C::NST));
        }
        __syncwarp();
      }
    }
    // every MMA issued is complete before the CTA leaves
    if (lane == 0) tc::mma_commit(bar_drain);
    mbar_wait_warp(bar_drain, 0, 1 << 20);
  } else if (warp >= kConvWarp0) {
    // ---------------------------------------------------------------- q8_0 / q4s tile conversion
    if constexpr (C::CONV) {
      constexpr int kItems = kT * 8 / (32 * kConvWarps);    // q8_0: 16-code chunks per thread and tile
      constexpr int kItems4 = kT * 4 / (32 * kConvWarps);   // q4s: 32-code blocks per thread and tile
      static_assert(kItems * 32 * kConvWarps == kT * 8 && kItems4 * 32 * kConvWarps == kT * 4, "converter items");
      const int ct = tid - 32 * kConvWarp0, nct = 32 * kConvWarps;
      ConvItem items[kItems];
      Conv4Item items4[kItems4];
#pragma unroll
      for (int u = 0; u < kItems; ++u) items[u] = conv_item(ct + nct * u);
#pragma unroll
      for (int u = 0; u < kItems4; ++u) items4[u] = conv4_item(ct + nct * u);
      for (int t = 0; t < n_tiles; ++t) {
        const int s = t % C::NST, bb = t & 1;
        if (!wait_phase(bar_full + 8 * s, (t / C::NST) & 1, abort_flag, wl)) break;
        const int nv = nv_of(t);
        const uint8_t* st = smem + s * C::STAGE;
        if constexpr (C::KQ) {
          if (t >= 2 && !wait_phase(kc_empty + 8 * bb, ((t >> 1) - 1) & 1, abort_flag, wl)) break;
          const int sg = tile_sigma(st + C::KSC_OFF, lane, nv);
          if constexpr (C::K4) convert_q4<kItems4>(st, st + C::KSC_OFF, smem + C::KC_OFF + bb * 2 * kTile16, items4, nv, sg);
          else convert_q8<kItems>(st, st + C::KSC_OFF, smem + C::KC_OFF + bb * 2 * kTile16, items, nv, sg);
          tc::fence_smem_to_async();
          warp_arrive(kc_full + 8 * bb, lane);
        }
        if constexpr (C::VQ) {
          if (t >= 2 && !wait_phase(vc_empty + 8 * bb, ((t >> 1) - 1) & 1, abort_flag, wl)) break;
          const int sg = tile_sigma(st + C::VSC_OFF, lane, nv);
          if constexpr (C::V4)
            convert_q4<kItems4>(st + C::V_OFF, st + C::VSC_OFF, smem + C::VC_OFF + bb * 2 * kTile16, items4, nv, sg);
          else convert_q8<kItems>(st + C::V_OFF, st + C::VSC_OFF, smem + C::VC_OFF + bb * 2 * kTile16, items, nv, sg);
          tc::fence_smem_to_async();
          warp_arrive(vc_full + 8 * bb, lane);
        }
        warp_arrive(bar_empty + 8 * s, lane);
      }
    }
  } else {
    // ---------------------------------------------------------------- softmax (warps 0-7)
    const int row = tid & (kRows - 1), half = warp >> 2;   // tensor-memory lane, score half
    const int r = row0 + row;
    const int lim = r < rows_total ? (int)(L - T + r / G) : -1;   // last position row r sees
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float* const red = reinterpret_cast<float*>(smem + C::RED_OFF);   // [tile & 1][half][row], sums
    // exchanges with the other warp of these rows: bounded mbarrier waits (an abort cannot
    // leave one of the two waiting for good)
    const uint32_t my_xch = xch + 24 * (warp & 3);
    // Q row, dims 64 half .. + 63 -> 16-bit pairs (f16; bf16 for a bf16 K) in tensor-memory
    // columns kColQ + 32 half ..
    {
      const bool qv = r < rows_total;
      const __nv_bfloat16* qrow =
          a.q + (((long long)b * T + (qv ? r / G : 0)) * a.num_q_heads + (long long)kvh * G + (qv ? r % G : 0)) * kD +
          64 * half;
      float w[32];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint4 x = make_uint4(0u, 0u, 0u, 0u);
        if (qv) x = *reinterpret_cast<const uint4*>(qrow + 8 * c);
        const float2 f0 = unpack2<true>(x.x), f1 = unpack2<true>(x.y), f2 = unpack2<true>(x.z),
                     f3 = unpack2<true>(x.w);
        w[4 * c + 0] = __uint_as_float(pack2<C::SBF>(f0.x, f0.y));   // bf16 Q for a bf16 K: as given
        w[4 * c + 1] = __uint_as_float(pack2<C::SBF>(f1.x, f1.y));
        w[4 * c + 2] = __uint_as_float(pack2<C::SBF>(f2.x, f2.y));
        w[4 * c + 3] = __uint_as_float(pack2<C::SBF>(f3.x, f3.y));
      }
      tc::tmem_st32(tmem + lane_off + kColQ + 32 * half, w);
      tc::fence_before_sync();
      warp_arrive(q_full, lane);
    }

    const int c0 = 32 * half;   // this thread's scores of a tile: columns c0 .. c0 + 31
    float m = -INFINITY, l = 0.0f;
    int sv_run = -1000;   // exponent of O's unit 2^-sv_run (q8_0 V)
    bool ok = true;
    for (int t = 0; t < n_tiles; ++t) {
      const int s = t % C::NST, bb = t & 1, pos0 = t * kT;
      // the tile's flags and prescale exponents, then the stage is this role's no more
      if (!wait_phase(bar_full + 8 * s, (t / C::NST) & 1, abort_flag, wl)) { ok = false; break; }
      const int nv = nv_of(t);
      const int sk = C::KQ ? tile_sigma(smem + s * C::STAGE + C::KSC_OFF, lane, nv) : 0;
      const int svt = C::VQ ? tile_sigma(smem + s * C::STAGE + C::VSC_OFF, lane, nv) : 0;
      if constexpr (!C::VQ) {
        // V rows past the length (or of a bad page) hold whatever the stage holds: zero them
        // before PV reads them (0 x NaN would reach O)
        if (nv < kT) {
          uint8_t* vt = smem + s * C::STAGE + C::V_OFF;
          for (int i = tid; i < (kT - nv) * 16; i += 32 * kSoftmaxWarps) {
            const int tt = nv + (i >> 4), c = i & 15;
            *reinterpret_cast<uint4*>(vt + tile_chunk(tt, c)) = make_uint4(0u, 0u, 0u, 0u);
          }
          tc::fence_smem_to_async();
        }
      }
      warp_arrive(bar_empty + 8 * s, lane);

      // scores of tile t (this thread's half)
      if (!wait_phase(s_full + 8 * bb, (t >> 1) & 1, abort_flag, wl)) { ok = false; break; }
      tc::fence_after_sync();
      float x[32];
      tc::tmem_ld32(tmem + lane_off + 64 * bb + c0, x);
      tc::fence_before_sync();
      warp_arrive(s_empty + 8 * bb, lane);

      // row maximum of the raw scores (mul > 0), masked entries -inf; four independent chains
      if (!(pos0 + c0 + 31 <= lim && c0 + 32 <= nv)) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (!(pos0 + c0 + j <= lim && c0 + j < nv)) x[j] = -INFINITY;
      }
      float mq[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
      for (int j = 4; j < 32; ++j) mq[j & 3] = fmaxf(mq[j & 3], x[j]);
      float mr = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
      red[(bb * 2 + half) * kRows + row] = mr;
      warp_arrive(my_xch + 8 * bb, lane);
      if (!wait_phase(my_xch + 8 * bb, (t >> 1) & 1, abort_flag, wl)) { ok = false; break; }
      mr = fmaxf(mr, red[(bb * 2 + (half ^ 1)) * kRows + row]);
      const float mul = a.qk_scale_log2 * __uint_as_float((uint32_t)(127 + sk) << 23);
      const float mx = mr * mul;

      const int sv_new = C::VQ ? max(sv_run, svt) : 0;
      float fo = 1.0f;   // this row's O rescale factor
      if (mx > m + kLazy || sv_new != sv_run) {
        const float nm = mx > m + kLazy ? mx : m;
        const float fm = m == -INFINITY ? 1.0f : fast_exp2(m - nm);
        // l is a sum of true p; O also carries the V tiles' unit 2^-sv_run
        l *= fm;
        m = nm;
        fo = fm * (C::VQ && sv_run > -1000 ? __uint_as_float((uint32_t)(127 + sv_run - sv_new) << 23) : 1.0f);
      }
      sv_run = sv_new;
      // O rescale (tensor-memory loads and stores are warp-wide: the warp's 32 rows together,
      // each by its own factor; this thread's 64 of the 128 columns) once PV(t - 1) is done
      if (__any_sync(0xffffffffu, t > 0 && fo != 1.0f)) {
        if (!wait_phase(p_empty + 8 * ((t - 1) & 1), ((t - 1) >> 1) & 1, abort_flag, wl)) { ok = false; break; }
        tc::fence_after_sync();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          float ov[32];
          tc::tmem_ld32(tmem + lane_off + kColO + 64 * half + 32 * c, ov);
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] *= fo;
          tc::tmem_st32(tmem + lane_off + kColO + 64 * half + 32 * c, ov);
        }
      }
      // PV takes p 2^(svt - sv_run) with p = 2^(s mul - m) (0 for masked entries and rows
      // that saw nothing): the power of two rides in the exponent, and l, a sum of true p,
      // takes the tile's sum times 2^(sv_run - svt) (exact)
      const float nb = (m == -INFINITY ? 0.0f : -m) + (C::VQ ? (float)(svt - sv_run) : 0.0f);
      float ph[16], pl[16];
      float2 ls[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
      for (int k = 0; k < 16; ++k) {
        const float2 e = __ffma2_rn(make_float2(x[2 * k], x[2 * k + 1]), make_float2(mul, mul), make_float2(nb, nb));
        const float2 p = make_float2(fast_exp2(e.x), fast_exp2(e.y));
        ls[k & 1] = __fadd2_rn(ls[k & 1], p);
        uint32_t h, lo;
        split2<C::PBF>(p.x, p.y, h, lo);
        ph[k] = __uint_as_float(h);
        pl[k] = __uint_as_float(lo);
      }
      const float lt = (ls[0].x + ls[1].x) + (ls[0].y + ls[1].y);
      l += C::VQ ? lt * __uint_as_float((uint32_t)(127 + sv_run - svt) << 23) : lt;
      // P buffer bb is free once PV(t - 2) is done
      if (t >= 2 && !wait_phase(p_empty + 8 * bb, ((t >> 1) - 1) & 1, abort_flag, wl)) { ok = false; break; }
      tc::fence_after_sync();
      tc::tmem_st16(tmem + lane_off + kColP + 64 * bb + 16 * half, ph);
      tc::tmem_st16(tmem + lane_off + kColP + 64 * bb + 32 + 16 * half, pl);
      tc::fence_before_sync();
      warp_arrive(p_full + 8 * bb, lane);
    }
    // O after the last PV; the row sum from both halves
    if (ok && n_tiles > 0) ok = wait_phase(p_empty + 8 * ((n_tiles - 1) & 1), ((n_tiles - 1) >> 1) & 1, abort_flag, wl);
    tc::fence_after_sync();
    red[(4 + half) * kRows + row] = l;
    warp_arrive(my_xch + 16, lane);
    if (!wait_phase(my_xch + 16, 0, abort_flag, wl)) ok = false;
    l += red[(4 + (half ^ 1)) * kRows + row];
    float* orow = r < rows_total
                      ? a.out + (((long long)b * T + r / G) * a.num_q_heads + (long long)kvh * G + r % G) * kD
                      : nullptr;
    const float inv = (ok && l > 0.0f && n_tiles > 0)
                          ? (C::VQ ? __uint_as_float((uint32_t)(127 + sv_run) << 23) : 1.0f) / l
                          : 0.0f;
#pragma unroll 1
    for (int c = 2 * half; c < 2 * half + 2; ++c) {
      float ov[32];
      tc::tmem_ld32(tmem + lane_off + kColO + 32 * c, ov);   // every lane: the load is warp-wide
      if (orow) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(orow + 32 * c + j) =
              inv != 0.0f ? make_float4(ov[j] * inv, ov[j + 1] * inv, ov[j + 2] * inv, ov[j + 3] * inv)
                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (tid == 0 && *abort_flag) record_fault(a.k.status, KVQ_DEVICE_TIMEOUT);
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int KC, int VC>
cudaError_t launch(const PrefillArgs& a, int batch, const CUtensorMap& tmk, const CUtensorMap& tmv,
                   cudaStream_t stream) {
  using C = TCfg<KC, VC>;
  auto kern = prefill_tc_kernel<KC, VC>;
  static unsigned long long done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!(dev < 64 && (done >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_RELAXED);
  }
  const int rows = a.tokens * a.group;
  const dim3 grid((unsigned)((rows + kRows - 1) / kRows), a.k.num_kv_heads, batch);
  e = launch_pdl(kern, grid, dim3(C::THREADS), C::SMEM, stream, tmk, tmv, a);
  count_launch();
  return e;
}

}  // namespace prefill_tc
}  // namespace kvq
