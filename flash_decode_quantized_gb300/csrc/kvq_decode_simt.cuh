// CUDA-core split-K flash-decode with dequantization fused into the QK^T and PV loops.
//
// The kernel class is the "flash-decode-over-quant" path that rMLX issue #292 (root
// cause, correction) identifies as the cost centre; the treatment is halobench record
// clm-0022's "dequantize KV on load": quantized K/V tiles are staged in shared memory
// as stored and converted to fp32 inside the dot products, never written back.
//
// Work split (step a2): grid = (n_chunks, num_kv_heads, batch).  A CTA owns one chunk of
// `chunk_tokens` consecutive tokens of one (sequence, KV head) and serves all G query
// heads of that KV head's group from the same tile (GQA sharing), so every KV byte is
// read from HBM once per decode.  Chunks past the sequence end exit at once.
//
// Per CTA (128 threads = 4 warps), per 32-token tile (steps a3..a6):
//   * cp.async 16-byte copies stage the tile's K rows, K scales, V rows and V scales
//     into shared memory, NS stages deep (rows padded by 16 bytes against bank
//     conflicts);
//   * QK^T: warp w takes tokens 8w..8w+7; a quad of lanes splits one token's head_dim
//     in four; each lane converts its stored elements to fp32 16 at a time and
//     accumulates q.k for every head of the group, applying the block scale d_k once
//     per 16 elements; a two-step shuffle finishes the dot product;
//   * online softmax per warp in base 2 (scores pre-multiplied by scale*log2(e)):
//     running max m and sum l per head, shuffle reductions over the warp's tokens;
//   * PV: lane l owns output elements [l*D/32, (l+1)*D/32) of every head; for each of
//     the warp's tokens it converts its V elements and accumulates p * d_v * v.
// After the chunk the four warps merge their (m, l, acc) in shared memory and write one
// partial per query head (step a7); a separate kernel combines the chunks (step a8).
#pragma once

#include "kvq_device.cuh"

namespace kvq {
namespace simt {

constexpr int kThreads = 128;
constexpr int kWarps = 4;
constexpr int kTileTokens = 32;
constexpr int kStages = 3;

template <int KC, int VC, int D, int GMAX>
struct Cfg {
  static constexpr int QD = D / 4;                  // dims per lane in QK^T
  static constexpr int EPL = D / 32;                // dims per lane in PV
  static constexpr int KRB = KC == KVQ_CODEC_Q8_0 ? D : KC == KVQ_CODEC_Q4S ? D / 2 : 2 * D;
  static constexpr int VRB = VC == KVQ_CODEC_Q8_0 ? D : VC == KVQ_CODEC_Q4S ? D / 2 : 2 * D;
  static constexpr int KNS = is_quant(KC) ? D / kBlock : 0;
  static constexpr int VNS = is_quant(VC) ? D / kBlock : 0;
  static constexpr int KPAD = KRB + 16;
  static constexpr int VPAD = VRB + 16;
  static constexpr int QROW = QD + 4;               // padded q quarter row (floats)
  // shared memory map (bytes)
  static constexpr int KQ_BYTES = kTileTokens * KPAD;
  static constexpr int KS_BYTES = ((kTileTokens * KNS * 2) + 15) / 16 * 16;
  static constexpr int VQ_BYTES = kTileTokens * VPAD;
  static constexpr int VS_BYTES = ((kTileTokens * VNS * 2) + 15) / 16 * 16;
  static constexpr int STAGE_BYTES = KQ_BYTES + KS_BYTES + VQ_BYTES + VS_BYTES;
  static constexpr int STAGES_BYTES = kStages * STAGE_BYTES;
  static constexpr int OBUF_BYTES = kWarps * GMAX * D * 4;
  static constexpr int UNION_BYTES = STAGES_BYTES > OBUF_BYTES ? STAGES_BYTES : OBUF_BYTES;
  static constexpr int QS_OFF = 0;
  static constexpr int QS_BYTES = GMAX * 4 * QROW * 4;
  static constexpr int PS_OFF = QS_OFF + QS_BYTES;
  static constexpr int PS_BYTES = kWarps * 8 * GMAX * 4;
  static constexpr int ML_OFF = PS_OFF + PS_BYTES;
  static constexpr int ML_BYTES = kWarps * GMAX * 2 * 4;
  static constexpr int UNION_OFF = (ML_OFF + ML_BYTES + 127) / 128 * 128;
  static constexpr int SMEM = UNION_OFF + UNION_BYTES;
};

template <int KC, int VC, int D, int GMAX>
__global__ void __launch_bounds__(kThreads, 2) decode_simt_kernel(DecodeArgs a) {
  using C = Cfg<KC, VC, D, GMAX>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* qs = reinterpret_cast<float*>(smem + C::QS_OFF);
  float* ps = reinterpret_cast<float*>(smem + C::PS_OFF);
  float* ml = reinterpret_cast<float*>(smem + C::ML_OFF);
  uint8_t* stages = smem + C::UNION_OFF;

  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = a.group;
  const int P = a.k.page_size;

  asm volatile("griddepcontrol.wait;" ::: "memory");   // no-op unless launched programmatically
  const long long cap = min((long long)a.max_pages * P, (long long)a.n_chunks * a.chunk_tokens);
  long long Lraw = a.seq_lens[b];
  if (Lraw < 0 || Lraw > cap) {
    if (tid == 0 && chunk == 0 && kvh == 0) {
      record_fault(a.k.status, KVQ_DEVICE_BAD_SEQ_LEN);
      record_fault(a.v.status, KVQ_DEVICE_BAD_SEQ_LEN);
    }
    Lraw = Lraw < 0 ? 0 : cap;
  }
  const int L = (int)Lraw;
  const int t_begin = chunk * a.chunk_tokens;
  if (t_begin >= L) return;
  const int t_end = min(L, t_begin + a.chunk_tokens);
  const int n_tiles = (t_end - t_begin + kTileTokens - 1) / kTileTokens;

  // q of the group, pre-scaled into base-2 logits, laid out [h][quarter][QROW].
  const __nv_bfloat16* qg = a.q + ((long long)b * a.num_q_heads + (long long)kvh * G) * D;
  for (int i = tid; i < GMAX * D; i += kThreads) {
    const int h = i / D, j = i % D;
    const float v = h < G ? __bfloat162float(qg[(long long)h * D + j]) * a.qk_scale_log2 : 0.0f;
    qs[(h * 4 + j / C::QD) * C::QROW + (j % C::QD)] = v;
  }

  const int32_t* pt = a.page_table + (long long)b * a.max_pages;
  auto tile_page = [&](int tile) -> int {
    const int pos0 = t_begin + tile * kTileTokens;
    return pt[pos0 / P];
  };
  auto page_ok = [&](int page) { return page >= 0 && page < a.k.num_pages && page < a.v.num_pages; };

  auto issue = [&](int tile, int stage) {
    const int pos0 = t_begin + tile * kTileTokens;
    const int row0 = pos0 % P;
    const int page = tile_page(tile);
    if (page_ok(page)) {
      uint8_t* st = stages + stage * C::STAGE_BYTES;
      const uint8_t* ks = a.k.buf + ((long long)page * a.k.num_kv_heads + kvh) * a.k.slab_bytes;
      const uint8_t* vs = a.v.buf + ((long long)page * a.v.num_kv_heads + kvh) * a.v.slab_bytes;
      constexpr int KCH = C::KRB / 16, VCH = C::VRB / 16;
      for (int i = tid; i < kTileTokens * KCH; i += kThreads) {
        const int r = i / KCH, c = i % KCH;
        cp_async16(st + r * C::KPAD + c * 16, ks + (long long)(row0 + r) * C::KRB + c * 16);
      }
      for (int i = tid; i < kTileTokens * VCH; i += kThreads) {
        const int r = i / VCH, c = i % VCH;
        cp_async16(st + C::KQ_BYTES + C::KS_BYTES + r * C::VPAD + c * 16,
                   vs + (long long)(row0 + r) * C::VRB + c * 16);
      }
      if constexpr (C::KNS > 0) {
        constexpr int N = kTileTokens * C::KNS * 2 / 16;
        const uint8_t* src = ks + (long long)P * C::KRB + (long long)row0 * C::KNS * 2;
        for (int i = tid; i < N; i += kThreads) cp_async16(st + C::KQ_BYTES + i * 16, src + i * 16);
      }
      if constexpr (C::VNS > 0) {
        constexpr int N = kTileTokens * C::VNS * 2 / 16;
        const uint8_t* src = vs + (long long)P * C::VRB + (long long)row0 * C::VNS * 2;
        for (int i = tid; i < N; i += kThreads)
          cp_async16(st + C::KQ_BYTES + C::KS_BYTES + C::VQ_BYTES + i * 16, src + i * 16);
      }
    } else if (tid == 0) {
      record_fault(a.k.status, KVQ_DEVICE_BAD_PAGE);
      record_fault(a.v.status, KVQ_DEVICE_BAD_PAGE);
    }
    cp_async_commit();
  };

  float m[GMAX], l[GMAX], acc[GMAX][C::EPL];
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int e = 0; e < C::EPL; ++e) acc[h][e] = 0.0f;
  }

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < n_tiles) issue(s, s);
    else cp_async_commit();
  }

  const int quarter = lane & 3;
  const int tok_w = lane >> 2;  // token within the warp's 8
  for (int tile = 0; tile < n_tiles; ++tile) {
    cp_async_wait<kStages - 2>();
    __syncthreads();
    {
      const int nt = tile + kStages - 1;
      if (nt < n_tiles) issue(nt, nt % kStages);
      else cp_async_commit();
    }
    const uint8_t* st = stages + (tile % kStages) * C::STAGE_BYTES;
    const int pos0 = t_begin + tile * kTileTokens;
    const bool tile_ok = page_ok(tile_page(tile));

    // ---- QK^T: this lane's quarter of token (8*warp + tok_w) against every head ----
    const int tl = warp * 8 + tok_w;
    const bool valid = tile_ok && (pos0 + tl < t_end);
    float s[GMAX];
#pragma unroll
    for (int h = 0; h < GMAX; ++h) s[h] = 0.0f;
    {
      const uint8_t* krow = st + tl * C::KPAD;
      const __half* ksc = reinterpret_cast<const __half*>(st + C::KQ_BYTES) + tl * C::KNS;
#pragma unroll
      for (int ch = 0; ch < C::QD / 16; ++ch) {
        const int e0 = quarter * C::QD + ch * 16;
        float kv[16];
        load16<KC>(krow + (long long)e0 * C::KRB / D, kv);
        float dk = 1.0f;
        if constexpr (C::KNS > 0) dk = __half2float(ksc[e0 / kBlock]);
#pragma unroll
        for (int h = 0; h < GMAX; ++h) {
          const float4* qv = reinterpret_cast<const float4*>(qs + (h * 4 + quarter) * C::QROW + ch * 16);
          float sb = 0.0f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 qq = qv[k];
            sb = fmaf(qq.x, kv[4 * k], sb);
            sb = fmaf(qq.y, kv[4 * k + 1], sb);
            sb = fmaf(qq.z, kv[4 * k + 2], sb);
            sb = fmaf(qq.w, kv[4 * k + 3], sb);
          }
          s[h] = fmaf(dk, sb, s[h]);
        }
      }
    }
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      s[h] += __shfl_xor_sync(0xffffffffu, s[h], 1);
      s[h] += __shfl_xor_sync(0xffffffffu, s[h], 2);
      if (!valid) s[h] = -INFINITY;
    }

    // ---- online softmax over the warp's 8 tokens (base 2) ----
    float* psw = ps + warp * 8 * GMAX;
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      float mx = s[h];
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m[h], mx);
      float alpha = 1.0f, p = 0.0f;
      if (m_new != -INFINITY) {
        alpha = fast_exp2(m[h] - m_new);
        p = fast_exp2(s[h] - m_new);
      }
      float sum = p;
      sum += __shfl_xor_sync(0xffffffffu, sum, 4);
      sum += __shfl_xor_sync(0xffffffffu, sum, 8);
      sum += __shfl_xor_sync(0xffffffffu, sum, 16);
      l[h] = fmaf(l[h], alpha, sum);
      m[h] = m_new;
#pragma unroll
      for (int e = 0; e < C::EPL; ++e) acc[h][e] *= alpha;
      if (quarter == 0) psw[tok_w * GMAX + h] = p;
    }
    __syncwarp();

    // ---- PV: lane owns elements [lane*EPL, (lane+1)*EPL) of every head ----
    const uint8_t* vq = st + C::KQ_BYTES + C::KS_BYTES;
    const __half* vsc = reinterpret_cast<const __half*>(st + C::KQ_BYTES + C::KS_BYTES + C::VQ_BYTES);
#pragma unroll 2
    for (int tt = 0; tt < 8; ++tt) {
      const int tok = warp * 8 + tt;
      if (!tile_ok || pos0 + tok >= t_end) break;  // tokens are in order: the rest are invalid too
      float vv[C::EPL];
      load_n<VC, C::EPL>(vq + tok * C::VPAD, lane * C::EPL, vv);
      float dv = 1.0f;
      if constexpr (C::VNS > 0) dv = __half2float(vsc[tok * C::VNS + (lane * C::EPL) / kBlock]);
#pragma unroll
      for (int h = 0; h < GMAX; ++h) {
        const float pd = psw[tt * GMAX + h] * dv;
#pragma unroll
        for (int e = 0; e < C::EPL; ++e) acc[h][e] = fmaf(pd, vv[e], acc[h][e]);
      }
    }
    __syncwarp();
  }

  // ---- merge the four warps' (m, l, acc) and write the chunk's partials (a7) ----
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  cp_async_wait<0>();
  __syncthreads();
  if (lane == 0) {
#pragma unroll
    for (int h = 0; h < GMAX; ++h) {
      ml[(warp * GMAX + h) * 2] = m[h];
      ml[(warp * GMAX + h) * 2 + 1] = l[h];
    }
  }
  __syncthreads();
  float* obuf = reinterpret_cast<float*>(stages);
#pragma unroll
  for (int h = 0; h < GMAX; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml[(w * GMAX + h) * 2]);
    const float sc = (m[h] == -INFINITY) ? 0.0f : fast_exp2(m[h] - M);
#pragma unroll
    for (int e = 0; e < C::EPL; ++e) obuf[(warp * GMAX + h) * D + lane * C::EPL + e] = acc[h][e] * sc;
  }
  __syncthreads();
  const long long head0 = (long long)b * a.num_q_heads + (long long)kvh * G;
  for (int i = tid; i < G * D; i += kThreads) {
    const int h = i / D, j = i % D;
    float o = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) o += obuf[(w * GMAX + h) * D + j];
    a.part_o[((head0 + h) * a.n_chunks + chunk) * D + j] = o;
  }
  for (int h = tid; h < G; h += kThreads) {
    float M = -INFINITY;
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, ml[(w * GMAX + h) * 2]);
    float lsum = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      const float mw = ml[(w * GMAX + h) * 2];
      if (mw != -INFINITY) lsum += fast_exp2(mw - M) * ml[(w * GMAX + h) * 2 + 1];
    }
    a.part_ml[((head0 + h) * a.n_chunks + chunk) * 2] = M;
    a.part_ml[((head0 + h) * a.n_chunks + chunk) * 2 + 1] = lsum;
  }
}

template <int KC, int VC, int D, int GMAX>
cudaError_t launch(const DecodeArgs& a, cudaStream_t stream) {
  using C = Cfg<KC, VC, D, GMAX>;
  auto kern = decode_simt_kernel<KC, VC, D, GMAX>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_chunks, a.k.num_kv_heads, a.batch);
  kern<<<grid, kThreads, C::SMEM, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

// Dispatch over head_dim and the group bound for one codec pair.
template <int KC, int VC>
cudaError_t launch_pair(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  const int g = a.group;
#define KVQ_SIMT_G(D)                                              \
  if (g <= 4) return launch<KC, VC, D, 4>(a, stream);              \
  if (g <= 8) return launch<KC, VC, D, 8>(a, stream);              \
  if (g <= 16) return launch<KC, VC, D, 16>(a, stream);            \
  return cudaErrorNotSupported;
  switch (head_dim) {
    case 64: { KVQ_SIMT_G(64) }
    case 128: { KVQ_SIMT_G(128) }
    case 256: { KVQ_SIMT_G(256) }
    default: return cudaErrorNotSupported;
  }
#undef KVQ_SIMT_G
}

}  // namespace simt
}  // namespace kvq
