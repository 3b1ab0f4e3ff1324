// Chunked prefill attention over the quantized store: T new tokens of a sequence (already
// appended, the last T positions) attend causally to everything before them and to each
// other, reading K and V straight from the paged quant store with the dequantization fused
// into the two contractions (the prompt-processing arm of halobench record clm-0022's
// depth tables, pp512 at depth, where dequantize-on-load also moved q8_0 prefill).
//
// Layout (query rows on M, as a prefill kernel wants them): a CTA owns 64 query rows of one
// KV head, row = token * G + head-in-group, 16 rows per warp.  Per 64-token KV tile:
//  * S = Q K^T: A = the warp's Q rows (registers, loaded once), B = the K tile.  Integer K
//    codes come from ldmatrix on the stored bytes and are turned into f16 in registers; the
//    k order inside a 16-element step follows the bytes each lane receives (Q is laid out
//    with the same permutation).  Each 32-element block accumulates into a fresh fragment
//    seeded with -offset * sum(q) of the block and is then scaled by that token's d_k.
//  * online softmax per row (base 2), the causal limit applied per element.
//  * O += P V: A = P scaled by the V block scale d_v[t, b] (per block, split hi + lo in the
//    16-bit type, with a running power-of-two bound of the scales keeping it in range),
//    B = the V tile via ldmatrix.trans, integer codes made exact f16 integers in registers.
// Tiles stream through the same TMA + mbarrier ring as the decode kernel; every wait is
// bounded.  No split over the KV length: a prompt has rows enough to fill the GPU.
#pragma once

#include "kvq_decode_mma.cuh"

namespace kvq {
namespace prefill {

using namespace kvq::mma;

constexpr int kRowsPerCta = 64;
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kPS = 14;   // P_b = p * d_v * 2^(kPS - E) <= 2^14 (p <= 1, d_v < 2^E)

template <int KC, int VC, int D>
struct PCfg {
  static constexpr bool KQ = is_quant(KC), VQ = is_quant(VC);
  static constexpr bool KBF = KC == KVQ_CODEC_BF16, VBF = VC == KVQ_CODEC_BF16;
  static constexpr int KRB = KC == KVQ_CODEC_Q8_0 ? D : KC == KVQ_CODEC_Q4S ? D / 2 : 2 * D;
  static constexpr int VRB = VC == KVQ_CODEC_Q8_0 ? D : VC == KVQ_CODEC_Q4S ? D / 2 : 2 * D;
  static constexpr int NB = D / kBlock;
  static constexpr int KSTEPS = D / 16;
  static constexpr int ONT = D / 8;                       // O n-tiles per warp
  static constexpr int al1k(int x) { return (x + 1023) / 1024 * 1024; }
  static constexpr int KROWS = al1k(kT * KRB), VROWS = al1k(kT * VRB);
  static constexpr int KSC = KQ ? kT * NB * 2 : 0, VSC = VQ ? kT * NB * 2 : 0;
  static constexpr int V_OFF = KROWS, KSC_OFF = KROWS + VROWS, VSC_OFF = KSC_OFF + KSC;
  static constexpr int STAGE = al1k(KROWS + VROWS + KSC + VSC);
  static constexpr int NS0 = (96 * 1024) / STAGE;
  static constexpr int NS = NS0 > 3 ? 3 : (NS0 < 2 ? 2 : NS0);
  static constexpr int BAR_OFF = NS * STAGE;
  static constexpr int OK_OFF = BAR_OFF + 2 * NS * 8;
  // head_dim 256: the warps' Q fragments live in shared memory ([warp][k-step][32 lanes] x 16
  // bytes) instead of registers, which the 16 x 256 O accumulators (128 per thread) need
  static constexpr bool QSM = D == 256;
  static constexpr int QF_OFF = OK_OFF + 32;
  // ... and the QK seeds ([warp][block][32 lanes] x float2)
  static constexpr int SD_OFF = QF_OFF + (QSM ? kWarps * KSTEPS * 512 : 0);
  static constexpr int SMEM = SD_OFF + (QSM ? kWarps * NB * 256 : 0) + 1024;
  static constexpr uint32_t K_TX = kT * KRB + KSC, V_TX = kT * VRB + VSC;
};

// Element of head_dim held by A-fragment k-slot `k` (0..15) of QK step `s`, matching the
// bytes ldmatrix hands lane quad i for each K codec (k = 2i, 2i+1, 2i+8, 2i+9 per lane).
template <int KC>
__device__ __forceinline__ int pf_qk_dim(int s, int k) {
  const int i = (k & 7) >> 1, e = k & 1, hi = k >> 3;
  if constexpr (KC == KVQ_CODEC_Q8_0) return 16 * s + 4 * i + 2 * hi + e;          // bytes 4i..4i+3
  else if constexpr (KC == KVQ_CODEC_Q4S) return 32 * (s >> 1) + 8 * i + 2 * (s & 1) + hi + 4 * e;
  else return 16 * s + 8 * hi + 2 * i + e;                                          // natural
}

template <int KC, int VC, int D>
__global__ void __launch_bounds__(kThreads)
prefill_mma_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   PrefillArgs a) {
  using C = PCfg<KC, VC, D>;
  extern __shared__ uint8_t smem_raw[];
  // (offset from the array itself, so accesses through `smem` stay in the shared space)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::BAR_OFF, bar_empty = sbase + C::BAR_OFF + 8 * C::NS;
  volatile int* stage_ok = reinterpret_cast<volatile int*>(smem + C::OK_OFF);

  const int rt = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, i4 = lane & 3;
  const int G = a.group, T = a.tokens;
  const int P = a.k.page_size;
  const int rows_total = T * G;
  const int row0 = rt * kRowsPerCta;

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
  // the CTA's last query token sees positions [0, L - T + i_last]
  const int i_last = min(row0 + kRowsPerCta - 1, rows_total - 1) / G;
  const long long kv_end_ll = min(L, L - T + i_last + 1);
  const int kv_end = kv_end_ll > 0 ? (int)kv_end_ll : 0;
  const int n_tiles = (kv_end + kT - 1) / kT;

  // rows of this lane: r_lo = warp*16 + g, r_hi = r_lo + 8; causal limits (last position)
  const int rA = row0 + warp * 16 + g, rB = rA + 8;
  const int limA = rA < rows_total ? (int)(L - T + rA / G) : -1;
  const int limB = rB < rows_total ? (int)(L - T + rB / G) : -1;

  if (tid == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, kWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

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
    const int s = tile % C::NS;
    const int pos0 = tile * kT;
    const int rr0 = pos0 % P;
    const uint32_t full = bar_full + 8 * s;
    const bool ok = page >= 0 && page < a.k.num_pages && page < a.v.num_pages;
    stage_ok[s] = ok ? 1 : 0;
    if (!ok) {
      record_fault(a.k.status, KVQ_DEVICE_BAD_PAGE);
      record_fault(a.v.status, KVQ_DEVICE_BAD_PAGE);
      mbar_arrive(full);
      return;
    }
    mbar_expect_tx(full, C::K_TX + C::V_TX);
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
  };
  if (warp == 0) {
    for (int tile = 0; tile < n_tiles && tile < C::NS; ++tile) {
      const int page = page_of(tile);
      if (lane == 0) issue_tile(tile, page);
    }
    __syncwarp();
  }

  // ---------------------------------------------------------------- Q fragments (A of QK)
  // (with QSM only the seeds keep them: the fragments go to shared memory below)
  uint32_t qa[C::KSTEPS][4];
  {
    const __nv_bfloat16* qrow[2];
    bool qv[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = h ? rB : rA;
      qv[h] = r < rows_total;
      const int tok = qv[h] ? r / G : 0, hh = qv[h] ? r % G : 0;
      qrow[h] = a.q + (((long long)b * T + tok) * a.num_q_heads + (long long)kvh * G + hh) * D;
    }
#pragma unroll
    for (int s = 0; s < C::KSTEPS; ++s) {
#pragma unroll
      for (int reg = 0; reg < 4; ++reg) {   // a0: row g, slots 2i..; a1: row g+8; a2/a3: slots 2i+8..
        const int h = reg & 1, hi = reg >> 1;
        const int k0 = 8 * hi + 2 * i4;
        const float x0 = qv[h] ? __bfloat162float(qrow[h][pf_qk_dim<KC>(s, k0)]) : 0.0f;
        const float x1 = qv[h] ? __bfloat162float(qrow[h][pf_qk_dim<KC>(s, k0 + 1)]) : 0.0f;
        qa[s][reg] = pack2<C::KBF>(x0, x1);
      }
    }
  }
  // QK accumulator seeds: -offset * (sum of the block's q as the MMA sees them), per row
  float seed[C::NB][2];
#pragma unroll
  for (int bb = 0; bb < C::NB; ++bb) {
    float sA = 0.0f, sB = 0.0f;
    if constexpr (C::KQ) {
#pragma unroll
      for (int s = 2 * bb; s < 2 * bb + 2; ++s) {
        const float2 f0 = unpack2<false>(qa[s][0]), f2 = unpack2<false>(qa[s][2]);
        const float2 f1 = unpack2<false>(qa[s][1]), f3 = unpack2<false>(qa[s][3]);
        sA += f0.x + f0.y + f2.x + f2.y;
        sB += f1.x + f1.y + f3.x + f3.y;
      }
      sA += __shfl_xor_sync(0xffffffffu, sA, 1);
      sA += __shfl_xor_sync(0xffffffffu, sA, 2);
      sB += __shfl_xor_sync(0xffffffffu, sB, 1);
      sB += __shfl_xor_sync(0xffffffffu, sB, 2);
    }
    const float bias = KC == KVQ_CODEC_Q4S ? kBias4K : kBias8;
    seed[bb][0] = -bias * sA;
    seed[bb][1] = -bias * sB;
  }
  const float qk_mul = a.qk_scale_log2 * (KC == KVQ_CODEC_Q4S ? kScale4K : 1.0f);
  uint4* const qfs = reinterpret_cast<uint4*>(smem + C::QF_OFF) + warp * C::KSTEPS * 32 + lane;
  float2* const sds = reinterpret_cast<float2*>(smem + C::SD_OFF) + warp * C::NB * 32 + lane;
  if constexpr (C::QSM) {
#pragma unroll
    for (int s = 0; s < C::KSTEPS; ++s) qfs[s * 32] = make_uint4(qa[s][0], qa[s][1], qa[s][2], qa[s][3]);
#pragma unroll
    for (int bb = 0; bb < C::NB; ++bb) sds[bb * 32] = make_float2(seed[bb][0], seed[bb][1]);
    __syncwarp();
  }
  // QK seeds of block bb (rows g, g + 8)
  auto seed_of = [&](int bb) -> float2 {
    if constexpr (C::QSM) return sds[bb * 32];
    else return make_float2(seed[bb][0], seed[bb][1]);
  };
  // A fragment of k-step ks
  auto qfrag = [&](int ks, uint32_t* f) {
    if constexpr (C::QSM) {
      const uint4 v = qfs[ks * 32];
      f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    } else {
      f[0] = qa[ks][0]; f[1] = qa[ks][1]; f[2] = qa[ks][2]; f[3] = qa[ks][3];
    }
  };

  float o[C::ONT][4];
#pragma unroll
  for (int n = 0; n < C::ONT; ++n)
#pragma unroll
    for (int k = 0; k < 4; ++k) o[n][k] = 0.0f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.0f, lB = 0.0f;
  int E = -100;   // running power-of-two bound of the V scales seen
  bool timed_out = false;
  const int mi = lane >> 3, mr = lane & 7;

  for (int tile = 0; tile < n_tiles; ++tile) {
    const int s = tile % C::NS;
    if (!mbar_wait_warp(bar_full + 8 * s, (tile / C::NS) & 1)) {
      timed_out = true;
      break;
    }
    const int pos0 = tile * kT;
    if (stage_ok[s] != 0) {
      const uint32_t st = sbase + s * C::STAGE;
      const uint32_t kst = st, vst = st + C::V_OFF;
      const uint8_t* ksc = smem + s * C::STAGE + C::KSC_OFF;
      const uint8_t* vsc = smem + s * C::STAGE + C::VSC_OFF;

      // ------------------------------------------------ S = Q K^T, [rows g, g+8] x [8 n-tiles]
      float sc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int k = 0; k < 4; ++k) sc[n][k] = 0.0f;
      if constexpr (C::KQ) {
#pragma unroll
        for (int nq = 0; nq < 2; ++nq) {       // n-tiles 4nq .. 4nq+3 (tokens 32nq .. +31)
#pragma unroll
          for (int bb = 0; bb < C::NB; ++bb) {
            float cb[4][4];
            const float2 sdb = seed_of(bb);
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              cb[m][0] = sdb.x; cb[m][1] = sdb.x;
              cb[m][2] = sdb.y; cb[m][3] = sdb.y;
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int ks = 2 * bb + half;
              uint32_t qk[4];
              qfrag(ks, qk);
              uint32_t y[4];
              // matrix m: tokens 8(4nq+m) .. +7; q8: chunk ks (16 dims); q4: chunk bb (32 dims)
              const int chunk = KC == KVQ_CODEC_Q8_0 ? ks : bb;
              ldsm_x4(row_chunk<C::KRB>(kst, 8 * (4 * nq + mi) + mr, chunk), y[0], y[1], y[2], y[3]);
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                uint32_t b0, b1;
                if constexpr (KC == KVQ_CODEC_Q8_0) {
                  const uint32_t u = y[m] ^ 0x80808080u;
                  b0 = i8pair_raw(u, 0x4140);
                  b1 = i8pair_raw(u, 0x4342);
                } else {
                  b0 = u4pair_half(half ? (y[m] >> 4) : (y[m] << 4));
                  b1 = u4pair_half(half ? (y[m] >> 8) : y[m]);
                }
                mma16816<false>(cb[m], qk, b0, b1);
              }
            }
            // scale by the tokens' block scales: columns 2*i4, 2*i4+1 of n-tile 4nq + m
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              const int n = 4 * nq + m;
              const int t0c = 8 * n + 2 * i4;
              const float d0 = __half2float(*reinterpret_cast<const __half*>(ksc + (t0c * C::NB + bb) * 2));
              const float d1 = __half2float(*reinterpret_cast<const __half*>(ksc + ((t0c + 1) * C::NB + bb) * 2));
              sc[n][0] = fmaf(d0, cb[m][0], sc[n][0]);
              sc[n][1] = fmaf(d1, cb[m][1], sc[n][1]);
              sc[n][2] = fmaf(d0, cb[m][2], sc[n][2]);
              sc[n][3] = fmaf(d1, cb[m][3], sc[n][3]);
            }
          }
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < C::KSTEPS; ++ks) {
          uint32_t qk[4];
          qfrag(ks, qk);
#pragma unroll
          for (int np = 0; np < 4; ++np) {   // n-tiles 2np, 2np+1: matrices (n, k lo), (n, k hi), ...
            uint32_t y[4];
            ldsm_x4(row_chunk<C::KRB>(kst, 8 * (2 * np + (mi >> 1)) + mr, 2 * ks + (mi & 1)), y[0], y[1], y[2], y[3]);
            mma16816<C::KBF>(sc[2 * np], qk, y[0], y[1]);
            mma16816<C::KBF>(sc[2 * np + 1], qk, y[2], y[3]);
          }
        }
      }

      // ------------------------------------------------ causal / length mask, online softmax
      float tmA = -INFINITY, tmB = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int p0 = pos0 + 8 * n + 2 * i4;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int p = p0 + (k & 1);
          const int lim = k < 2 ? limA : limB;
          float v = sc[n][k] * qk_mul;
          if (p > lim || p >= kv_end) v = -INFINITY;
          sc[n][k] = v;
        }
        tmA = fmaxf(tmA, fmaxf(sc[n][0], sc[n][1]));
        tmB = fmaxf(tmB, fmaxf(sc[n][2], sc[n][3]));
      }
      tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 1));
      tmA = fmaxf(tmA, __shfl_xor_sync(0xffffffffu, tmA, 2));
      tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 1));
      tmB = fmaxf(tmB, __shfl_xor_sync(0xffffffffu, tmB, 2));

      // V-scale bound of the tile (warp-uniform): every d_v of the tile is < 2^Et
      int Et = -127;
      if constexpr (C::VQ) {
        uint32_t mx = 0;   // scales of the tile's tokens below kv_end (rows past it are stale)
        for (int w = lane; w < kT * C::NB / 2; w += 32)
          if (pos0 + w / (C::NB / 2) < kv_end) mx = __vmaxu2(mx, reinterpret_cast<const uint32_t*>(vsc)[w]);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) mx = __vmaxu2(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const uint32_t hmax = max(mx & 0xffffu, mx >> 16);
        Et = hmax ? max((int)(hmax >> 10), 1) - 14 : -127;
      } else {
        Et = 0;   // 16-bit V: no scale, P <= 1
      }
      const int E_new = max(E, Et);
      const float newA = fmaxf(mA, tmA), newB = fmaxf(mB, tmB);
      const float e2 = __uint_as_float((uint32_t)(127 + E - E_new) << 23);   // 2^(E - E_new)
      const float fA = (newA == -INFINITY) ? 1.0f : fast_exp2(mA - newA);
      const float fB = (newB == -INFINITY) ? 1.0f : fast_exp2(mB - newB);
      lA *= fA;
      lB *= fB;
      if (fA != 1.0f || fB != 1.0f || E_new != E) {
        const float gA = fA * e2, gB = fB * e2;
#pragma unroll
        for (int n = 0; n < C::ONT; ++n) {
          o[n][0] *= gA; o[n][1] *= gA; o[n][2] *= gB; o[n][3] *= gB;
        }
      }
      mA = newA; mB = newB; E = E_new;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        sc[n][0] = sc[n][0] == -INFINITY ? 0.0f : fast_exp2(sc[n][0] - mA);
        sc[n][1] = sc[n][1] == -INFINITY ? 0.0f : fast_exp2(sc[n][1] - mA);
        sc[n][2] = sc[n][2] == -INFINITY ? 0.0f : fast_exp2(sc[n][2] - mB);
        sc[n][3] = sc[n][3] == -INFINITY ? 0.0f : fast_exp2(sc[n][3] - mB);
        lA += sc[n][0] + sc[n][1];
        lB += sc[n][2] + sc[n][3];
      }

      // ------------------------------------------------ O += P V
      const float pscale = C::VQ ? __uint_as_float((uint32_t)(127 + kPS - E) << 23) : 1.0f;
#pragma unroll
      for (int kk = 0; kk < kT / 16; ++kk) {
        // P of tokens 16kk + {2i, 2i+1} (n-tile 2kk) and 16kk + 8 + {2i, 2i+1} (n-tile 2kk+1)
        const float* p_lo = sc[2 * kk];
        const float* p_hi = sc[2 * kk + 1];
        if constexpr (C::VQ) {
#pragma unroll
          for (int bb = 0; bb < C::NB; ++bb) {
            const int tt = 16 * kk + 2 * i4;
            const float dv0 = __half2float(*reinterpret_cast<const __half*>(vsc + (tt * C::NB + bb) * 2)) * pscale;
            const float dv1 = __half2float(*reinterpret_cast<const __half*>(vsc + ((tt + 1) * C::NB + bb) * 2)) * pscale;
            const float dv8 = __half2float(*reinterpret_cast<const __half*>(vsc + ((tt + 8) * C::NB + bb) * 2)) * pscale;
            const float dv9 = __half2float(*reinterpret_cast<const __half*>(vsc + ((tt + 9) * C::NB + bb) * 2)) * pscale;
            uint32_t ah[4], al[4];
            split2<false>(p_lo[0] * dv0, p_lo[1] * dv1, ah[0], al[0]);   // row g, tokens 2i, 2i+1
            split2<false>(p_lo[2] * dv0, p_lo[3] * dv1, ah[1], al[1]);   // row g+8
            split2<false>(p_hi[0] * dv8, p_hi[1] * dv9, ah[2], al[2]);   // row g, tokens 8+2i, 8+2i+1
            split2<false>(p_hi[2] * dv8, p_hi[3] * dv9, ah[3], al[3]);   // row g+8
            if constexpr (VC == KVQ_CODEC_Q8_0) {
              // matrices: (tok 0-7, chunk 2b), (tok 8-15, chunk 2b), (tok 0-7, 2b+1), (tok 8-15, 2b+1)
              uint32_t y[4];
              ldsm_x4_t(row_chunk<C::VRB>(vst, 16 * kk + 8 * (mi & 1) + mr, 2 * bb + (mi >> 1)), y[0], y[1], y[2], y[3]);
#pragma unroll
              for (int c = 0; c < 2; ++c) {        // 16-dim chunk 2b + c
                const uint32_t ulo = y[2 * c] ^ 0x80808080u, uhi = y[2 * c + 1] ^ 0x80808080u;
#pragma unroll
                for (int par = 0; par < 2; ++par) {   // dims 16(2b+c) + 2n + par
                  const uint32_t sel = par ? 0x4341 : 0x4240;
                  const uint32_t b0 = hsub2_u32(i8pair_raw(ulo, sel), 0x64806480u);
                  const uint32_t b1 = hsub2_u32(i8pair_raw(uhi, sel), 0x64806480u);
                  float* acc = o[2 * (2 * bb + c) + par];
                  mma16816<false>(acc, ah, b0, b1);
                  mma16816<false>(acc, al, b0, b1);
                }
              }
            } else {   // q4s: one 16-byte chunk per block; the lane gets 4 nibbles of 2 tokens
              uint32_t y[2];
              {
                uint32_t y2, y3;
                // matrices: (tok 0-7, chunk b), (tok 8-15, chunk b), repeated (x4 needs 4 addresses)
                ldsm_x4_t(row_chunk<C::VRB>(vst, 16 * kk + 8 * (mi & 1) + mr, bb), y[0], y[1], y2, y3);
              }
              // y: [t 2i: nibbles 4n..4n+3 (dims 4n+e)][t 2i+1: same dims], n = g (16-bit col g)
#pragma unroll
              for (int e = 0; e < 4; ++e) {   // dims 4n + e of the block
                // even nibbles: 1024 + u, less 1032; odd nibbles in place: (1024 + 16 u) / 16 - 72
                const int sh = 4 * (e & ~1);
                const uint32_t b0 = (e & 1) ? hfma2_u32(u4pair_hi_raw(y[0] >> sh), kSixteenth2, kMinus72x2)
                                            : hsub2_u32(u4pair_raw(y[0] >> sh), 0x64086408u);
                const uint32_t b1 = (e & 1) ? hfma2_u32(u4pair_hi_raw(y[1] >> sh), kSixteenth2, kMinus72x2)
                                            : hsub2_u32(u4pair_raw(y[1] >> sh), 0x64086408u);
                float* acc = o[4 * bb + e];
                mma16816<false>(acc, ah, b0, b1);
                mma16816<false>(acc, al, b0, b1);
              }
            }
          }
        } else {
          uint32_t ah[4], al[4];
          split2<C::VBF>(p_lo[0], p_lo[1], ah[0], al[0]);
          split2<C::VBF>(p_lo[2], p_lo[3], ah[1], al[1]);
          split2<C::VBF>(p_hi[0], p_hi[1], ah[2], al[2]);
          split2<C::VBF>(p_hi[2], p_hi[3], ah[3], al[3]);
#pragma unroll
          for (int np = 0; np < C::ONT / 2; ++np) {
            // matrices: (tok 0-7, dims 16np..+7), (tok 8-15, same), (tok 0-7, 16np+8..), (tok 8-15, ..)
            uint32_t y[4];
            ldsm_x4_t(row_chunk<C::VRB>(vst, 16 * kk + 8 * (mi & 1) + mr, 2 * np + (mi >> 1)), y[0], y[1], y[2], y[3]);
            mma16816<C::VBF>(o[2 * np], ah, y[0], y[1]);
            mma16816<C::VBF>(o[2 * np], al, y[0], y[1]);
            mma16816<C::VBF>(o[2 * np + 1], ah, y[2], y[3]);
            mma16816<C::VBF>(o[2 * np + 1], al, y[2], y[3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    if (warp == 0 && tile + C::NS < n_tiles) {
      if (!mbar_wait_warp(bar_empty + 8 * s, (tile / C::NS) & 1)) {
        timed_out = true;
        break;
      }
      const int page = page_of(tile + C::NS);
      if (lane == 0) issue_tile(tile + C::NS, page);
      __syncwarp();
    }
  }
  if (timed_out) record_fault(a.k.status, KVQ_DEVICE_TIMEOUT);

  // ---------------------------------------------------------------- normalize and write
  lA += __shfl_xor_sync(0xffffffffu, lA, 1);
  lA += __shfl_xor_sync(0xffffffffu, lA, 2);
  lB += __shfl_xor_sync(0xffffffffu, lB, 1);
  lB += __shfl_xor_sync(0xffffffffu, lB, 2);
  const float oscale = C::VQ ? __uint_as_float((uint32_t)(127 + E - kPS) << 23) : 1.0f;
  const float invA = lA > 0.0f ? oscale / lA : 0.0f, invB = lB > 0.0f ? oscale / lB : 0.0f;
  float* outA = nullptr;
  float* outB = nullptr;
  if (rA < rows_total) outA = a.out + (((long long)b * T + rA / G) * a.num_q_heads + (long long)kvh * G + rA % G) * D;
  if (rB < rows_total) outB = a.out + (((long long)b * T + rB / G) * a.num_q_heads + (long long)kvh * G + rB % G) * D;
#pragma unroll
  for (int n = 0; n < C::ONT; ++n) {
    // columns 2*i4, 2*i4+1 of O n-tile n -> head_dim elements
    int d0, d1;
    if constexpr (VC == KVQ_CODEC_Q8_0) {
      const int chunk = n >> 1, par = n & 1;          // dims 16*chunk + 2*col + par
      d0 = 16 * chunk + 4 * i4 + par;
      d1 = d0 + 2;
    } else if constexpr (VC == KVQ_CODEC_Q4S) {
      const int blk = n >> 2, e = n & 3;              // dims 32*blk + 4*col + e
      d0 = 32 * blk + 8 * i4 + e;
      d1 = d0 + 4;
    } else {
      d0 = 8 * n + 2 * i4;
      d1 = d0 + 1;
    }
    if (outA) { outA[d0] = o[n][0] * invA; outA[d1] = o[n][1] * invA; }
    if (outB) { outB[d0] = o[n][2] * invB; outB[d1] = o[n][3] * invB; }
  }
}

template <int KC, int VC, int D>
cudaError_t launch(const PrefillArgs& a, int batch, const CUtensorMap& tmk, const CUtensorMap& tmv,
                   cudaStream_t stream) {
  using C = PCfg<KC, VC, D>;
  auto kern = prefill_mma_kernel<KC, VC, D>;
  static unsigned long long done = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!(dev < 64 && (done >> dev) & 1ull)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev < 64) __atomic_fetch_or(&done, 1ull << dev, __ATOMIC_RELAXED);
  }
  const int rows = a.tokens * a.group;
  const dim3 grid((unsigned)((rows + kRowsPerCta - 1) / kRowsPerCta), a.k.num_kv_heads, batch);
  e = launch_pdl(kern, grid, dim3(kThreads), C::SMEM, stream, tmk, tmv, a);
  count_launch();
  return e;
}

template <int KC, int VC>
cudaError_t launch_pair(const PrefillArgs& a, int batch, int head_dim, const CUtensorMap& tmk,
                        const CUtensorMap& tmv, cudaStream_t stream) {
  switch (head_dim) {
    case 64: return launch<KC, VC, 64>(a, batch, tmk, tmv, stream);
    case 128: return launch<KC, VC, 128>(a, batch, tmk, tmv, stream);
    case 256: return launch<KC, VC, 256>(a, batch, tmk, tmv, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace prefill
}  // namespace kvq
