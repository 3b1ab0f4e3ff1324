// Chunked prefill attention on the 5th-generation tensor cores (tcgen05, accumulators in
// tensor memory), head_dim 128, K and V each q8_0 or f16: the prompt-processing arm of
// halobench record clm-0022's depth tables (pp512 at depth), with the dequantization fused
// into the load of each KV tile.
//
// A CTA owns 128 query rows of one (sequence, KV head), row = token * G + head-in-group;
// thread t owns row t and tensor-memory lane t.  Per 64-token KV tile:
//  * the tile arrives by TMA in the 128-byte swizzled layout that the MMA reads; a q8_0 tile
//    is first turned, once for all 128 rows, into two f16 tiles of the same layout whose sum
//    is d * q exactly (hi = d q rounded, lo = the rounding error, exact in f16: d has 11
//    significant bits and q 7), with a power of two 2^-sigma folded in per tile (from the
//    tile's largest scale) that keeps every hi below 2^15;
//  * S = Q K^T: M 128 x N 64 x K 128 (two MMAs per K step for a q8_0 K: hi and lo) into 64
//    tensor-memory columns; S is exact up to the f32 sums, as in the 16-bit path;
//  * softmax by row (each thread its own row; base 2, lazy running maximum as in the decode
//    kernels); P is written to shared memory as f16 hi + lo (P = P_h + P_l to ~22 bits);
//  * O += P V: M 128 x N 128 x K 64, V as an MN-major operand straight from the tile layout;
//    P_h V_h + P_l V_h (+ P_h V_l for a q8_0 V), O in 128 tensor-memory columns.  A q8_0 V
//    tile carries its own 2^-sigma; O is kept in units of the largest sigma so far and
//    rescaled (with the lazy maximum's rescale) when it grows.
// Each step waits for the previous one (one tile in flight on the tensor cores); every wait
// is bounded and a timeout is reported in the K store's status word.
#pragma once

#include "kvq_decode_mma.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace prefill_tc {

using namespace kvq::mma;

constexpr int kD = 128;
constexpr int kRows = 128;        // query rows per CTA = threads = tensor-memory lanes
constexpr int kThreads = 128;
constexpr int kStages = 3;
constexpr int kTmemCols = 256;    // S: columns 0..63, O: columns 128..255
constexpr int kTile16 = kT * kD * 2;   // one 64 x 128 f16 operand tile (16 KB)

template <int KC, int VC>
struct TCfg {
  static constexpr bool KQ = KC == KVQ_CODEC_Q8_0, VQ = VC == KVQ_CODEC_Q8_0;
  static constexpr int NB = kD / kBlock;
  static constexpr int KRB = KQ ? kD : 2 * kD, VRB = VQ ? kD : 2 * kD;
  static constexpr int KROWS = kT * KRB, VROWS = kT * VRB;
  static constexpr int KSC = KQ ? kT * NB * 2 : 0, VSC = VQ ? kT * NB * 2 : 0;
  static constexpr int V_OFF = KROWS, KSC_OFF = KROWS + VROWS, VSC_OFF = KSC_OFF + KSC;
  static constexpr int al1k(int x) { return (x + 1023) / 1024 * 1024; }
  static constexpr int STAGE = al1k(KROWS + VROWS + KSC + VSC);
  static constexpr int KH_OFF = kStages * STAGE;                 // converted K: hi, lo
  static constexpr int VH_OFF = KH_OFF + (KQ ? 2 * kTile16 : 0);  // converted V: hi, lo
  static constexpr int Q_OFF = VH_OFF + (VQ ? 2 * kTile16 : 0);   // Q: 128 rows x 128 f16
  static constexpr int P_OFF = Q_OFF + kRows * kD * 2;            // P hi, P lo: 128 x 64 f16 each
  static constexpr int BAR_OFF = P_OFF + 2 * kRows * kT * 2;      // full[kStages], s_done, o_done
  static constexpr int MISC_OFF = BAR_OFF + 8 * (kStages + 2);    // tensor-memory base, stage flags
  static constexpr int SMEM = MISC_OFF + 64 + 1024;
  static constexpr uint32_t TX = KROWS + VROWS + KSC + VSC;
  static_assert(SMEM <= 227 * 1024, "shared memory");
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

// q8_0 tile (TMA layout, one 128-byte line per row) + its scales -> f16 hi and lo tiles of
// the two-region layout, d q 2^-sigma = hi + lo exactly; rows >= n_valid become zeros.
__device__ __forceinline__ void convert_q8(const uint8_t* rows, const uint8_t* sc, uint8_t* dst, int tid,
                                           int n_valid, int sigma) {
  const float f = __uint_as_float((uint32_t)(127 - sigma) << 23);
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int i = tid + kThreads * u, t = i >> 3, c = i & 7;   // row, 16-code chunk
    uint32_t hi[8], lo[8];
    if (t < n_valid) {
      const uint4 w = *reinterpret_cast<const uint4*>(rows + t * 128 + (((c ^ (t & 7)) << 4)));
      const float d = __half2float(*reinterpret_cast<const __half*>(sc + (t * 4 + (c >> 1)) * 2)) * f;
      const uint32_t d2 = pack2<false>(d, d);
      const uint32_t ws[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u, w.w ^ 0x80808080u};
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t q2 = hsub2_u32(i8pair_raw(ws[k >> 1], (k & 1) ? 0x4342 : 0x4140), 0x64806480u);
        __half2 h = __hmul2(*reinterpret_cast<const __half2*>(&q2), *reinterpret_cast<const __half2*>(&d2));
        hi[k] = *reinterpret_cast<uint32_t*>(&h);
        const uint32_t nh = hi[k] ^ 0x80008000u;
        lo[k] = hfma2_u32(q2, d2, nh);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) hi[k] = lo[k] = 0u;
    }
    const int oc = 2 * c;   // f16 chunks 2c, 2c + 1 of the row (dims 16 c .. 16 c + 15)
    *reinterpret_cast<uint4*>(dst + tile_chunk(t, oc)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(dst + tile_chunk(t, oc + 1)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    *reinterpret_cast<uint4*>(dst + kTile16 + tile_chunk(t, oc)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(dst + kTile16 + tile_chunk(t, oc + 1)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
  }
}

template <int KC, int VC>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  PrefillArgs a) {
  using C = TCfg<KC, VC>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::BAR_OFF, bar_s = bar_full + 8 * kStages, bar_o = bar_s + 8;
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
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
  const int r = row0 + tid;
  const int lim = r < rows_total ? (int)(L - T + r / G) : -1;   // last position row r sees

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(bar_full + 8 * s, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) tc::tmem_alloc(sbase + C::MISC_OFF, kTmemCols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = misc[0];
  const uint32_t t_s = tmem, t_o = tmem + 128;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  // ---------------------------------------------------------------- producer (warp 0)
  auto load_page = [&](int tile) -> int {
    const long long pos0 = (long long)tile * kT;
    return pos0 < cap ? __ldg(pt + pos0 / P) : -1;
  };
  int pg_lo = -1, pg_hi = -1, pb = 0;
  if (warp == 0) {
    pg_lo = load_page(lane);
    pg_hi = load_page(32 + lane);
  }
  auto page_of = [&](int t) -> int {
    while (t >= pb + 32) {
      pg_lo = pg_hi;
      pb += 32;
      pg_hi = load_page(pb + 32 + lane);
    }
    return __shfl_sync(0xffffffffu, pg_lo, t - pb);
  };
  auto issue_tile = [&](int tile, int page) {   // lane 0 of warp 0
    const int s = tile % kStages;
    const int rr0 = (tile * kT) % P;
    const uint32_t full = bar_full + 8 * s;
    const bool ok = page >= 0 && page < a.k.num_pages && page < a.v.num_pages;
    stage_ok[s] = ok ? 1 : 0;
    if (!ok) {
      record_fault(a.k.status, KVQ_DEVICE_BAD_PAGE);
      record_fault(a.v.status, KVQ_DEVICE_BAD_PAGE);
      mbar_arrive(full);
      return;
    }
    mbar_expect_tx(full, C::TX);
    const uint32_t st = sbase + s * C::STAGE;
#pragma unroll
    for (int seg = 0; seg < C::KRB / 128; ++seg) tma_load_4d(st + seg * kT * 128, &tmk, seg * 128, rr0, kvh, page, full);
#pragma unroll
    for (int seg = 0; seg < C::VRB / 128; ++seg)
      tma_load_4d(st + C::V_OFF + seg * kT * 128, &tmv, seg * 128, rr0, kvh, page, full);
    if constexpr (C::KQ)
      bulk_load(st + C::KSC_OFF, a.k.buf + ((long long)page * a.k.num_kv_heads + kvh) * a.k.slab_bytes +
                                     (long long)P * C::KRB + (long long)rr0 * C::NB * 2,
                kT * C::NB * 2, full);
    if constexpr (C::VQ)
      bulk_load(st + C::VSC_OFF, a.v.buf + ((long long)page * a.v.num_kv_heads + kvh) * a.v.slab_bytes +
                                     (long long)P * C::VRB + (long long)rr0 * C::NB * 2,
                kT * C::NB * 2, full);
  };
  if (warp == 0) {
    for (int tile = 0; tile < n_tiles && tile < kStages; ++tile) {
      const int page = page_of(tile);
      if (lane == 0) issue_tile(tile, page);
    }
    __syncwarp();
  }
  int issued = min(n_tiles, kStages);

  // ---------------------------------------------------------------- Q row -> f16 operand
  {
    const bool qv = r < rows_total;
    const __nv_bfloat16* qrow =
        a.q + (((long long)b * T + (qv ? r / G : 0)) * a.num_q_heads + (long long)kvh * G + (qv ? r % G : 0)) * kD;
    uint8_t* qs = smem + C::Q_OFF;
#pragma unroll 4
    for (int c = 0; c < kD / 8; ++c) {
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (qv) {
        const uint4 x = *reinterpret_cast<const uint4*>(qrow + 8 * c);
        const float2 f0 = unpack2<true>(x.x), f1 = unpack2<true>(x.y), f2 = unpack2<true>(x.z), f3 = unpack2<true>(x.w);
        w = make_uint4(pack2<false>(f0.x, f0.y), pack2<false>(f1.x, f1.y), pack2<false>(f2.x, f2.y),
                       pack2<false>(f3.x, f3.y));
      }
      *reinterpret_cast<uint4*>(qs + (c >> 3) * (kRows * 128) + tid * 128 + (((c & 7) ^ (tid & 7)) << 4)) = w;
    }
  }

  const uint32_t idS = tc::idesc_f16(kRows, kT, false), idO = tc::idesc_f16(kRows, kD, true);
  const uint32_t sQ = sbase + C::Q_OFF, sPh = sbase + C::P_OFF, sPl = sPh + kRows * kT * 2;
  uint8_t* const ph_row = smem + C::P_OFF + tid * 128;
  uint8_t* const pl_row = ph_row + kRows * kT * 2;
  float m = -INFINITY, l = 0.0f;
  int sv_run = -1000;          // exponent of O's unit 2^-sv_run (q8_0 V)
  int n_s = 0, n_o = 0;        // S and PV rounds committed
  bool o_pending = false, timed_out = false;

  int tile = 0;
  for (; tile < n_tiles; ++tile) {
    const int s = tile % kStages;
    const uint32_t st = sbase + s * C::STAGE;
    bool ok = true;
    if (o_pending) {   // the previous PV round is done: P, the operand tiles and O are free
      ok = mbar_wait_warp(bar_o, (n_o - 1) & 1);
      o_pending = !ok;
    }
    ok = mbar_wait_warp(bar_full + 8 * s, (tile / kStages) & 1) && ok;
    if (__syncthreads_or(!ok)) {
      timed_out = true;
      break;
    }
    tc::fence_after_sync();
    // refill the stage of the previous tile (its data are converted or read by finished MMAs)
    if (tile > 0 && issued < n_tiles) {
      if (warp == 0) {
        const int page = page_of(issued);
        if (lane == 0) issue_tile(issued, page);
        __syncwarp();
      }
      ++issued;
    }
    if (stage_ok[s] == 0) continue;
    const int pos0 = tile * kT;
    const int n_valid = min(kT, kv_end - pos0);

    // ---------------------------------------------------------------- operand tiles
    int sk = 0, svt = 0;
    uint32_t kb = st, vb = st + C::V_OFF;
    if constexpr (C::KQ) {
      sk = tile_sigma(smem + s * C::STAGE + C::KSC_OFF, lane, n_valid);
      convert_q8(smem + s * C::STAGE, smem + s * C::STAGE + C::KSC_OFF, smem + C::KH_OFF, tid, n_valid, sk);
      kb = sbase + C::KH_OFF;
    }
    if constexpr (C::VQ) {
      svt = tile_sigma(smem + s * C::STAGE + C::VSC_OFF, lane, n_valid);
      convert_q8(smem + s * C::STAGE + C::V_OFF, smem + s * C::STAGE + C::VSC_OFF, smem + C::VH_OFF, tid, n_valid,
                 svt);
      vb = sbase + C::VH_OFF;
    } else if (n_valid < kT) {
      // rows past the length hold whatever the page holds: zero them (0 x NaN would reach O)
      uint8_t* vt = smem + s * C::STAGE + C::V_OFF;
      for (int i = tid; i < (kT - n_valid) * 16; i += kThreads) {
        const int t = n_valid + (i >> 4), c = i & 15;
        *reinterpret_cast<uint4*>(vt + tile_chunk(t, c)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------------------------------------------------------- S = Q K^T
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kD / 16; ++ks) {
        const uint64_t ad = tc::sdesc_sw128(sQ + (ks >> 2) * (kRows * 128) + (ks & 3) * 32, 16, 1024);
        const uint64_t bd = tc::sdesc_sw128(kb + (ks >> 2) * (kT * 128) + (ks & 3) * 32, 16, 1024);
        tc::mma_f16(t_s, ad, bd, idS, ks > 0);
        if constexpr (C::KQ) {
          const uint64_t bl = tc::sdesc_sw128(kb + kTile16 + (ks >> 2) * (kT * 128) + (ks & 3) * 32, 16, 1024);
          tc::mma_f16(t_s, ad, bl, idS, true);
        }
      }
      tc::mma_commit(bar_s);
    }
    ++n_s;
    if (__syncthreads_or(!mbar_wait_warp(bar_s, (n_s - 1) & 1))) {
      timed_out = true;
      break;
    }
    tc::fence_after_sync();

    // ---------------------------------------------------------------- softmax of this row
    float x[kT];
    tc::tmem_ld32(t_s + lane_off, x);
    tc::tmem_ld32(t_s + lane_off + 32, x + 32);
    const float mul = a.qk_scale_log2 * __uint_as_float((uint32_t)(127 + sk) << 23);
    float mx = -INFINITY;
    if (pos0 + kT - 1 <= lim) {
#pragma unroll
      for (int j = 0; j < kT; ++j) {
        x[j] *= mul;
        mx = fmaxf(mx, x[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < kT; ++j) {
        x[j] = pos0 + j <= lim ? x[j] * mul : -INFINITY;
        mx = fmaxf(mx, x[j]);
      }
    }
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
    // tensor-memory loads and stores are warp-wide (.sync.aligned): a warp rescales its 32
    // rows together, each by its own factor (1 where nothing moved)
    if (__any_sync(0xffffffffu, n_o > 0 && fo != 1.0f)) {
#pragma unroll 1
      for (int c = 0; c < kD / 32; ++c) {
        float ov[32];
        tc::tmem_ld32(t_o + lane_off + 32 * c, ov);
#pragma unroll
        for (int j = 0; j < 32; ++j) ov[j] *= fo;
        tc::tmem_st32(t_o + lane_off + 32 * c, ov);
      }
    }
    // p = 2^(x - m) (0 for masked entries and rows that saw nothing); the MMA takes p 2^(svt - sv_run)
    const float base = m == -INFINITY ? 0.0f : m;
    const float vsc = C::VQ ? __uint_as_float((uint32_t)(127 + svt - sv_run) << 23) : 1.0f;
    float lsum = 0.0f;
#pragma unroll
    for (int c = 0; c < kT / 8; ++c) {
      uint32_t h[4], lo4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float p0 = fast_exp2(x[8 * c + 2 * k] - base), p1 = fast_exp2(x[8 * c + 2 * k + 1] - base);
        lsum += p0 + p1;
        split2<false>(p0 * vsc, p1 * vsc, h[k], lo4[k]);
      }
      const uint32_t co = (uint32_t)(((c ^ (tid & 7)) << 4));
      *reinterpret_cast<uint4*>(ph_row + co) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(pl_row + co) = make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]);
    }
    l += lsum;
    tc::fence_smem_to_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // ---------------------------------------------------------------- O += P V
    if (tid == 0) {
#pragma unroll
      for (int kk = 0; kk < kT / 16; ++kk) {
        const uint64_t ah = tc::sdesc_sw128(sPh + kk * 32, 16, 1024);
        const uint64_t al = tc::sdesc_sw128(sPl + kk * 32, 16, 1024);
        const uint64_t bh = tc::sdesc_sw128(vb + kk * 2048, kT * 128, 1024);
        tc::mma_f16(t_o, ah, bh, idO, n_o > 0 || kk > 0);
        tc::mma_f16(t_o, al, bh, idO, true);
        if constexpr (C::VQ) {
          const uint64_t bl = tc::sdesc_sw128(vb + kTile16 + kk * 2048, kT * 128, 1024);
          tc::mma_f16(t_o, ah, bl, idO, true);
        }
      }
      tc::mma_commit(bar_o);
    }
    ++n_o;
    o_pending = true;
  }

  // ---------------------------------------------------------------- drain, normalize, write
  if (o_pending && !mbar_wait_warp(bar_o, (n_o - 1) & 1)) timed_out = true;
  if (__syncthreads_or(timed_out)) {
    // stages still being filled: wait (bounded) so that no copy lands after the CTA leaves
    for (int t = tile; t < issued; ++t) mbar_wait_warp(bar_full + 8 * (t % kStages), (t / kStages) & 1, 1 << 16);
    if (tid == 0) record_fault(a.k.status, KVQ_DEVICE_TIMEOUT);
  }
  tc::fence_after_sync();
  {
    // every lane takes part in the (warp-wide) tensor-memory loads; rows past the chunk store nothing
    float* orow = r < rows_total
                      ? a.out + (((long long)b * T + r / G) * a.num_q_heads + (long long)kvh * G + r % G) * kD
                      : nullptr;
    const float inv = (l > 0.0f && n_o > 0)
                          ? (C::VQ ? __uint_as_float((uint32_t)(127 + sv_run) << 23) : 1.0f) / l
                          : 0.0f;
#pragma unroll 1
    for (int c = 0; c < kD / 32; ++c) {
      float ov[32];
      tc::tmem_ld32(t_o + lane_off + 32 * c, ov);
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
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
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
  e = launch_pdl(kern, grid, dim3(kThreads), C::SMEM, stream, tmk, tmv, a);
  count_launch();
  return e;
}

}  // namespace prefill_tc
}  // namespace kvq
