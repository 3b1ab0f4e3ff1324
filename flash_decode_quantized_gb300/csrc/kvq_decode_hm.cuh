// Tensor-core decode, "heads on M" tile loop: for groups of 9 to 32 query rows per KV head
// (GQA 16:1, or fewer heads times several query tokens), included by kvq_decode_mma.cuh.
//
// With 16 or more query rows per KV head the rows fill the M dimension of mma.sync
// m16n8k16 by themselves, so both contractions put them there (16 rows per head group)
// and every K and V code of a tile is converted once per head group rather than once per
// 8-head group as in the tokens-on-M loop:
//
//  * QK^T: S[h, t] = sum_b d_k[t, b] * sum_{j in b} q[h, j] * k_int[t, j]
//    (halobench record clm-0022, "dequantize KV on load"; the q8_0 block layout of rMLX
//    issue #292).  A = q (16 rows x 16 elements per k-step, in shared memory in fragment
//    order), B = the stored K rows of 8 tokens read with ldmatrix: each lane gets 4
//    consecutive codes of one token, turned into the f16 pair (1152 + k) by a byte
//    permute; the element order inside a k-step is permuted to match those bytes and q is
//    laid out with the same permutation.  Each block's two k-steps start from the seed
//    -1152 * sum_{j in b} q[h, j] and are scaled by d_k[t, b] afterwards.
//  * PV: O[h, j] += sum_t P_b[h, t] * v_int[t, j] with P_b = p * d_v[t, b] * 2^(kPScale - E),
//    split into f16 hi and lo parts (two MMAs on the same B operand) so that the products
//    keep fp32-level accuracy.  The S accumulators of the slice's two 8-token N-tiles are
//    the A fragment of the 16-token k-step as they stand (no transpose).  B = V rows read
//    with ldmatrix.trans: the even and odd elements of a 16-element chunk form two N-tiles,
//    converted to exact f16 integers.
//
// Each warp takes 16 tokens of every 64-token tile for 16 query rows; the softmax state
// (running max in log2 units, lazily raised, and the sum) is per row, held by the quad of
// lanes that owns the row.  The tile producer, the ring of stages and the split-K combine
// are those of the tokens-on-M loop.
#pragma once

namespace kvq {
namespace mma {

// q of this CTA's KV head for the heads-on-M loop: loaded into registers at the start of
// the kernel (in flight together with the page-table and length reads), then stored to
// shared memory in MMA A-fragment order, with the QK seeds, once the first tiles are
// issued.  Nothing here when the loop is not in use.
template <int KC, int D, int HG, int THREADS, bool ON>
struct HmQ {
  __device__ __forceinline__ void load(const DecodeArgs&, long long, int) {}
};
template <int KC, int D, int HG, int THREADS>
struct HmQ<KC, D, HG, THREADS, true> {
  static_assert(KC == KVQ_CODEC_Q8_0, "heads-on-M loop: q8_0 K");
  static constexpr int QS = D / 16, NB = D / 32;
  static constexpr int NE = (HG * QS * 32 + THREADS - 1) / THREADS;   // fragment entries per thread
  static constexpr int NSD = (HG * NB * 16 + THREADS - 1) / THREADS;  // seeds per thread
  uint32_t w[NE][4];      // bf16 pairs of the entries
  uint4 sq[NSD][4];       // the 32 bf16 of each seed's (row, block)

  // Entry (group g, k-step s, lane (r, c)): a0 (row r, k 2c), a1 (row r + 8, k 2c),
  // a2 (row r, k 2c + 8), a3 (row r + 8, k 2c + 8).  For q8_0 K the pair (k, k + 1)
  // holds head_dim elements 16 s + 4c + 2 (k >= 8) + {0, 1}: one aligned 32-bit load.
  __device__ __forceinline__ void load(const DecodeArgs& a, long long row0, int G) {
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const int idx = threadIdx.x + e * THREADS;
      const int l = idx & 31, st = (idx >> 5) % QS, g = idx / (32 * QS);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int v = 16 * g + (l >> 2) + 8 * (j & 1);
        w[e][j] = 0u;
        if (idx < HG * QS * 32 && v < G)
          w[e][j] = __ldg(reinterpret_cast<const uint32_t*>(a.q + (row0 + v) * D + 16 * st + 4 * (l & 3) + 2 * (j >> 1)));
      }
    }
#pragma unroll
    for (int e = 0; e < NSD; ++e) {
      const int idx = threadIdx.x + e * THREADS;
      const int row = idx & 15, bb = (idx >> 4) % NB, g = idx / (16 * NB);
      const int v = 16 * g + row;
#pragma unroll
      for (int k = 0; k < 4; ++k) sq[e][k] = make_uint4(0u, 0u, 0u, 0u);
      if (idx < HG * NB * 16 && v < G) {
        const uint4* src = reinterpret_cast<const uint4*>(a.q + (row0 + v) * D + 32 * bb);
#pragma unroll
        for (int k = 0; k < 4; ++k) sq[e][k] = __ldg(src + k);
      }
    }
  }
  static __device__ __forceinline__ uint32_t bf2_to_h2(uint32_t x) {
    return pack2<false>(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
  }
  // fragments [HG][QS][32] x 16 bytes; seeds [HG][NB][8] x float4 (row r, row r, row r + 8,
  // row r + 8), the QK accumulator's initial value: -1152 times the sum of the block's q as
  // the f16 values the MMA multiplies
  __device__ __forceinline__ void store(uint8_t* smem_qf, uint8_t* smem_sd) const {
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      const int idx = threadIdx.x + e * THREADS;
      if (idx < HG * QS * 32)
        reinterpret_cast<uint4*>(smem_qf)[idx] =
            make_uint4(bf2_to_h2(w[e][0]), bf2_to_h2(w[e][1]), bf2_to_h2(w[e][2]), bf2_to_h2(w[e][3]));
    }
#pragma unroll
    for (int e = 0; e < NSD; ++e) {
      const int idx = threadIdx.x + e * THREADS;
      if (idx >= HG * NB * 16) continue;
      const int row = idx & 15, bb = (idx >> 4) % NB, g = idx / (16 * NB);
      float sum = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t x[4] = {sq[e][k].x, sq[e][k].y, sq[e][k].z, sq[e][k].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float2 f = unpack2<false>(bf2_to_h2(x[u]));
          sum += f.x + f.y;
        }
      }
      const float sv = -kBias8 * sum;
      reinterpret_cast<float2*>(smem_sd)[((g * NB + bb) * 8 + (row & 7)) * 2 + (row >> 3)] = make_float2(sv, sv);
    }
  }
};

// The tile loop of one warp and the CTA's merge of its warps.  Returns true when the CTA
// wrote a split-K partial for the in-place combine (the caller then runs it), false when
// it wrote the output itself or leaves its partial to the chunk merge kernel.
template <int KC, int VC, int D, int GW, int HG, class QRegs, class IssueFn, class PageFn, class TicketFn>
__device__ __forceinline__ bool hm_body(const DecodeArgs& a, uint8_t* smem, int b, int kvh, int chunk, int pipe,
                                        int pw, int warp, int lane, int tid, int vchunk, int nvc, int n_tiles,
                                        int L, int nv, uint32_t sring, uint32_t bar_full, uint32_t bar_empty,
                                        volatile int* stage_ok, const int* pgs, unsigned* rcnt,
                                        volatile int* last_issued, IssueFn& issue_tile, PageFn& load_page,
                                        bool take_ticket, TicketFn& ticket, const QRegs& hmq) {
  using C = Cfg<KC, VC, D, GW, HG>;
  static_assert(KC == KVQ_CODEC_Q8_0 && VC == KVQ_CODEC_Q8_0, "heads-on-M loop: q8_0 K and V");
  constexpr int QS = D / 16, NB = D / 32, NT8 = D / 8;
  const int G = a.group, T = a.tokens;
  const long long head0 = (long long)b * a.num_q_heads + (long long)kvh * G;
  const int NWT = C::NW * 32;
  const int hg = pw >> 2, ws = pw & 3;               // head group, 16-token slice

  hmq.store(smem + C::QF_OFF, smem + C::SD_OFF);
  asm volatile("bar.sync 1, %0;" ::"r"(C::THREADS) : "memory");
  // fused advance: the CTA's ticket, taken after the last CTA-wide barrier before the loop
  if (take_ticket && warp == C::NW - 1 && lane == 0) ticket();

  const int t0 = ws * 16;
  const int r = lane >> 2, c = lane & 3;
  const int mi = lane >> 3, mr = lane & 7;            // ldmatrix address roles
  const uint4* qf = reinterpret_cast<const uint4*>(smem + C::QF_OFF) + hg * QS * 32 + lane;
  const float4* sdp = reinterpret_cast<const float4*>(smem + C::SD_OFF) + hg * NB * 8 + r;
  uint8_t* const ring = smem + pipe * C::PRING;
  const int va = 16 * hg + r, vb = va + 8;           // this lane's rows (virtual heads)
  const int lim_a = L - T + 1 + va % T, lim_b = L - T + 1 + vb % T;   // causal limits (T > 1)
  // the slice's block scales as f32: K [NB][16 tokens], then V [NB][16 tokens]
  float* const scw = reinterpret_cast<float*>(smem + C::SC_OFF) + warp * 2 * NB * 16;
  // Per-lane byte offsets of the ldmatrix rows inside a stage's K or V rows (128-byte
  // swizzle: 16-byte chunk x of row t sits at (x >> 3) * 64 * 128 + t * 128 + ((x ^ t) & 7) * 16,
  // and t & 7 = mr for every row a lane addresses): row t0 + 8 (mi >> 1) + mr, chunk
  // 2 bb + (mi & 1), one offset per bb & 3
  uint32_t roff[4];
#pragma unroll
  for (int e = 0; e < 4; ++e)
    roff[e] = (t0 + 8 * (mi >> 1) + mr) * 128 + ((((2 * e + (mi & 1)) ^ mr) & 7) << 4);
  static_assert(C::KRB == D && C::VRB == D && D >= 128, "q8_0 rows of at least 128 bytes");

  float o[NT8][4];   // O N-tile j = 4 * block + 2 * chunk + parity
#pragma unroll
  for (int j = 0; j < NT8; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) o[j][k] = 0.0f;
  // running max of rows r, r + 8 (log2 units), and their sums and O in units of
  // 2^(E - kPScale) (E: running power-of-two bound of this warp's V scales)
  float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.0f, l_b = 0.0f;
  int E = -100;
  const float qk_mul = a.qk_scale_log2;
  bool timed_out = false;
  const int wlim = a.wait_limit;

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
      const uint32_t kst = sring + s * C::STAGE, vst = kst + C::V_OFF;
      const uint8_t* ksc = ring + s * C::STAGE + C::KSC_OFF;
      const uint8_t* vsc = ring + s * C::STAGE + C::VSC_OFF;

      // ---------------- block scales to f32: lane (t, h) converts blocks h NB/2 .. of token
      // t; V scales of tokens past the end are zeroed (their stage bytes are not data), which
      // also keeps them out of E
      uint32_t vmax = 0u;   // largest V scale bit pattern seen by this lane (scales are >= 0)
      {
        constexpr int PL = NB / 2;                     // values per lane (2 lanes per token)
        const int tt = lane >> 1, b0 = (lane & 1) * PL;
        uint32_t kw[PL / 2], vw[PL / 2];
#pragma unroll
        for (int u = 0; u < PL / 2; ++u) {
          kw[u] = *reinterpret_cast<const uint32_t*>(ksc + (t0 + tt) * NB * 2 + (b0 + 2 * u) * 2);
          vw[u] = *reinterpret_cast<const uint32_t*>(vsc + (t0 + tt) * NB * 2 + (b0 + 2 * u) * 2);
        }
#pragma unroll
        for (int u = 0; u < PL / 2; ++u) {
          const float2 f = unpack2<false>(kw[u]);
          scw[(b0 + 2 * u) * 16 + tt] = f.x;
          scw[(b0 + 2 * u + 1) * 16 + tt] = f.y;
        }
        const bool tv = tt < n_valid;
#pragma unroll
        for (int u = 0; u < PL / 2; ++u) {
          const uint32_t x = tv ? vw[u] : 0u;
          vmax = max(vmax, max(x & 0xffffu, x >> 16));
          const float2 f = unpack2<false>(x);
          scw[(NB + b0 + 2 * u) * 16 + tt] = f.x;
          scw[(NB + b0 + 2 * u + 1) * 16 + tt] = f.y;
        }
      }
      __syncwarp();
      const uint32_t vmax_w = __reduce_max_sync(0xffffffffu, vmax);
      const int ex_w = vmax_w ? max((int)(vmax_w >> 10), 1) - 14 : -127;   // this warp's V scales < 2^ex_w

      // ---------------- QK^T: S (unscaled) as pairs: sc[nt][0] rows r, sc[nt][1] rows r + 8,
      // columns tokens 8 nt + 2c, 8 nt + 2c + 1
      float2 sc[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = make_float2(0.0f, 0.0f);
#pragma unroll
      for (int bb = 0; bb < NB; ++bb) {
        uint32_t w0, w1, w2, w3;
        // matrices: (tok 0-7, chunk 2bb), (tok 0-7, chunk 2bb+1), (tok 8-15, 2bb), (tok 8-15, 2bb+1)
        ldsm_x4(kst + roff[bb & 3] + (bb >> 2) * (kT * 128), w0, w1, w2, w3);
        w0 ^= 0x80808080u; w1 ^= 0x80808080u; w2 ^= 0x80808080u; w3 ^= 0x80808080u;
        const uint4 qa = qf[(2 * bb) * 32], qb = qf[(2 * bb + 1) * 32];
        const uint32_t fa[4] = {qa.x, qa.y, qa.z, qa.w}, fb[4] = {qb.x, qb.y, qb.z, qb.w};
        float cb[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float4 sd = sdp[bb * 8];
          cb[nt][0] = sd.x; cb[nt][1] = sd.y; cb[nt][2] = sd.z; cb[nt][3] = sd.w;
        }
        // first k-steps of both N-tiles, then second k-steps
        mma16816<false>(cb[0], fa, i8pair_raw(w0, 0x4140), i8pair_raw(w0, 0x4342));
        mma16816<false>(cb[1], fa, i8pair_raw(w2, 0x4140), i8pair_raw(w2, 0x4342));
        mma16816<false>(cb[0], fb, i8pair_raw(w1, 0x4140), i8pair_raw(w1, 0x4342));
        mma16816<false>(cb[1], fb, i8pair_raw(w3, 0x4140), i8pair_raw(w3, 0x4342));
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          // tokens 8 nt + 2c, 8 nt + 2c + 1: S += d_k * block dot, as f32 pairs
          const float2 dk = *reinterpret_cast<const float2*>(scw + bb * 16 + 8 * nt + 2 * c);
          sc[nt][0] = __ffma2_rn(dk, make_float2(cb[nt][0], cb[nt][1]), sc[nt][0]);
          sc[nt][1] = __ffma2_rn(dk, make_float2(cb[nt][2], cb[nt][3]), sc[nt][1]);
        }
      }
      if (n_valid < 16 || (T > 1 && pos_w + 16 > L - T + 1)) {
        // tokens past the end, and the causal limit of each query token
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const int tok = 8 * nt + 2 * c, lim = hr ? lim_b : lim_a;
            float2& x = sc[nt][hr];
            if (tok >= n_valid || pos_w + tok >= lim) x.x = -INFINITY;
            if (tok + 1 >= n_valid || pos_w + tok + 1 >= lim) x.y = -INFINITY;
          }
      }

      // ---------------- lazy online softmax, per row.  Scores in log2 units are s * qk_mul
      // (qk_mul > 0).
      const float lma = fmaxf(fmaxf(sc[0][0].x, sc[0][0].y), fmaxf(sc[1][0].x, sc[1][0].y)) * qk_mul;
      const float lmb = fmaxf(fmaxf(sc[0][1].x, sc[0][1].y), fmaxf(sc[1][1].x, sc[1][1].y)) * qk_mul;
      const bool over = (lma > m_a + kLazy) || (lmb > m_b + kLazy) || (ex_w > E);
      if (__any_sync(0xffffffffu, over)) {
        float xa = lma, xb2 = lmb;
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
          xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, off));
          xb2 = fmaxf(xb2, __shfl_xor_sync(0xffffffffu, xb2, off));
        }
        const int E_new = max(E, ex_w);
        // the reference max of a row moves only past the lazy margin
        const float na = xa > m_a + kLazy ? fmaxf(m_a, xa) : m_a;
        const float nb = xb2 > m_b + kLazy ? fmaxf(m_b, xb2) : m_b;
        const float e2 = __uint_as_float((uint32_t)(127 + E - E_new) << 23);  // 2^(E - E_new)
        const float fa = ((na == -INFINITY) ? 1.0f : fast_exp2(m_a - na)) * e2;
        const float fb = ((nb == -INFINITY) ? 1.0f : fast_exp2(m_b - nb)) * e2;
        l_a *= fa;
        l_b *= fb;
#pragma unroll
        for (int j = 0; j < NT8; ++j) {
          o[j][0] *= fa; o[j][1] *= fa; o[j][2] *= fb; o[j][3] *= fb;
        }
        m_a = na;
        m_b = nb;
        E = E_new;
      }
      // p * 2^(kPScale - E) = 2^(s qk_mul - m + kPScale - E); a row whose every score so far
      // was masked keeps m = -inf and its p are 0
      const float ba = (float)(kPScale - E) - (m_a == -INFINITY ? 0.0f : m_a);
      const float bb2 = (float)(kPScale - E) - (m_b == -INFINITY ? 0.0f : m_b);
      float2 p[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        p[nt][0] = make_float2(fast_exp2(fmaf(sc[nt][0].x, qk_mul, ba)), fast_exp2(fmaf(sc[nt][0].y, qk_mul, ba)));
        p[nt][1] = make_float2(fast_exp2(fmaf(sc[nt][1].x, qk_mul, bb2)), fast_exp2(fmaf(sc[nt][1].y, qk_mul, bb2)));
      }
      l_a += (p[0][0].x + p[0][0].y) + (p[1][0].x + p[1][0].y);
      l_b += (p[0][1].x + p[0][1].y) + (p[1][1].x + p[1][1].y);

      // ---------------- PV, block by block
#pragma unroll
      for (int bb = 0; bb < NB; ++bb) {
        // A fragment: a0 (row r, tok 2c | 2c+1), a1 (row r+8, ...), a2 (row r, tok 2c+8 | 2c+9), a3
        uint32_t ahi[4], alo[4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float2 dv = *reinterpret_cast<const float2*>(scw + (NB + bb) * 16 + 8 * nt + 2 * c);
          const float2 pa = __fmul2_rn(p[nt][0], dv);
          const float2 pb = __fmul2_rn(p[nt][1], dv);
          split2<false>(pa.x, pa.y, ahi[2 * nt], alo[2 * nt]);
          split2<false>(pb.x, pb.y, ahi[2 * nt + 1], alo[2 * nt + 1]);
        }
        uint32_t y0, y1, y2, y3;
        // matrices: (tok 0-7, chunk 2bb), (tok 0-7, chunk 2bb+1), (tok 8-15, 2bb), (tok 8-15, 2bb+1)
        ldsm_x4_t(vst + roff[bb & 3] + (bb >> 2) * (kT * 128), y0, y1, y2, y3);
        // B fragments of the block's four N-tiles (chunk h, even / odd elements): the
        // even elements 2n of a chunk are bytes 0, 2 of each word, the odd ones bytes 1, 3
        uint32_t bv[4][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t ya = (h ? y1 : y0) ^ 0x80808080u, yb = (h ? y3 : y2) ^ 0x80808080u;
          bv[2 * h][0] = hsub2_u32(i8pair_raw(ya, 0x4240), 0x64806480u);
          bv[2 * h][1] = hsub2_u32(i8pair_raw(yb, 0x4240), 0x64806480u);
          bv[2 * h + 1][0] = hsub2_u32(i8pair_raw(ya, 0x4341), 0x64806480u);
          bv[2 * h + 1][1] = hsub2_u32(i8pair_raw(yb, 0x4341), 0x64806480u);
        }
        // hi parts into the four accumulators, then lo parts (no accumulator twice in a row)
#pragma unroll
        for (int n = 0; n < 4; ++n) mma16816<false>(o[4 * bb + n], ahi, bv[n][0], bv[n][1]);
#pragma unroll
        for (int n = 0; n < 4; ++n) mma16816<false>(o[4 * bb + n], alo, bv[n][0], bv[n][1]);
      }
    }
    // release the stage; the pipeline's last warp to release it refills it
    __syncwarp();
    const bool last = release_last(bar_empty + 8 * s, rcnt + s, lane, C::PW);
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

  // ------------------------------------------------------------ merge the warps
  if (timed_out) {
    record_fault(a.k.status, KVQ_DEVICE_TIMEOUT);
    // no bulk copy left in flight: wait for the last tile issued into each stage
    for (int st = 0; st < C::NS; ++st) {
      const int t = last_issued[st];
      if (t >= 0) (void)mbar_wait_warp(bar_full + 8 * st, (t / C::NS) & 1);
    }
  }
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    l_a += __shfl_xor_sync(0xffffffffu, l_a, off);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, off);
  }
  const float oscale = __uint_as_float((uint32_t)(127 + E - kPScale) << 23);   // true scale of l and O
  float2* mlw = reinterpret_cast<float2*>(smem + C::ML_OFF);      // [NW][16] (m, l) per row
  float2* hml = mlw + C::NW * 16;                                 // [HG * 16] (M, l) of the CTA
  if (c == 0) {
    mlw[warp * 16 + r] = make_float2(m_a, l_a * oscale);
    mlw[warp * 16 + r + 8] = make_float2(m_b, l_b * oscale);
  }
  // every warp reaches this barrier (a timed-out warp skips only its tiles); after it all
  // loops are done, so the rings are idle
  asm volatile("bar.sync 1, %0;" ::"r"(NWT) : "memory");
  // warps of head group g: pipeline pp, slice w -> warp pp * PW + 4 g + w (i = 4 pp + w)
  constexpr int GWARPS = 4 * C::NP;
  auto gwarp = [&](int g, int i) { return (i >> 2) * C::PW + 4 * g + (i & 3); };
  float Ma = -INFINITY, Mb = -INFINITY;
#pragma unroll
  for (int i = 0; i < GWARPS; ++i) {
    Ma = fmaxf(Ma, mlw[gwarp(hg, i) * 16 + r].x);
    Mb = fmaxf(Mb, mlw[gwarp(hg, i) * 16 + r + 8].x);
  }
  if (ws == 0 && (warp / C::PW) == 0 && c < 2) {
    // the CTA's sum for row r (c = 0) or r + 8 (c = 1) of this head group
    const int row = r + 8 * c;
    const float M = c ? Mb : Ma;
    float lsum = 0.0f;
    for (int i = 0; i < GWARPS; ++i) {
      const float2 x = mlw[gwarp(hg, i) * 16 + row];
      if (x.x != -INFINITY) lsum += fast_exp2(x.x - M) * x.y;
    }
    hml[16 * hg + row] = make_float2(M, lsum);
  }
  {
    // this warp's O in register order, scaled to the CTA maximum (one float4 per lane and
    // N-tile: rows r (k = 0, 1) and r + 8 (k = 2, 3))
    const float fa = (m_a == -INFINITY) ? 0.0f : fast_exp2(m_a - Ma) * oscale;
    const float fb = (m_b == -INFINITY) ? 0.0f : fast_exp2(m_b - Mb) * oscale;
    float4* ob = reinterpret_cast<float4*>(smem) + warp * NT8 * 32 + lane;
#pragma unroll
    for (int j = 0; j < NT8; ++j) ob[j * 32] = make_float4(o[j][0] * fa, o[j][1] * fa, o[j][2] * fb, o[j][3] * fb);
  }
  asm volatile("bar.sync 1, %0;" ::"r"(NWT) : "memory");
  // Output float4 (group g, row half rh, block bb, chunk h, lane (r, c)): row r + 8 rh, elements
  // 32 bb + 16 h + 4c .. + 3 of head_dim, which are (k = 2 rh, 2 rh + 1) of the even N-tile
  // j = 4 bb + 2 h and of the odd one j + 1 (elements 4c, 4c + 2 and 4c + 1, 4c + 3)
  const float2* obuf = reinterpret_cast<const float2*>(smem);
  const bool direct = nv == 1 && !a.chunk_merge;   // the whole sequence is this chunk
  for (int t = tid; t < HG * 2 * (NT8 / 2) * 32; t += NWT) {
    const int ln = t & 31, rest = t >> 5;
    const int jp = rest % (NT8 / 2), rh = (rest / (NT8 / 2)) & 1, g = rest / NT8;
    const int row = (ln >> 2) + 8 * rh, v = 16 * g + row;
    if (v >= G) continue;
    const int j = 2 * jp;
    float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < GWARPS; ++i) {
      const int w = gwarp(g, i);
      const float2 e = obuf[((w * NT8 + j) * 32 + ln) * 2 + rh];
      const float2 od = obuf[((w * NT8 + j + 1) * 32 + ln) * 2 + rh];
      sum.x += e.x; sum.y += od.x; sum.z += e.y; sum.w += od.y;
    }
    const int dim = 16 * jp + 4 * (ln & 3);
    if (direct) {
      const float lsum = hml[v].y;
      const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
      *reinterpret_cast<float4*>(a.out + (head0 + v) * D + dim) =
          make_float4(sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv);
    } else {
      *reinterpret_cast<float4*>(a.part_o + ((head0 + v) * a.n_chunks + chunk) * D + dim) = sum;   // a7
    }
  }
  if (direct) return false;
  for (int v = tid; v < G && v < 16 * HG; v += NWT)
    reinterpret_cast<float2*>(a.part_ml)[(head0 + v) * a.n_chunks + chunk] = hml[v];
  // with the chunk merge kernel the combine is that kernel's
  return !a.chunk_merge;
}

}  // namespace mma
}  // namespace kvq
