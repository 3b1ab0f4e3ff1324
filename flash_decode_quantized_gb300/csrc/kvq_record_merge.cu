// Split-K combines (step a8) launched after the tensor-core decode kernel: the record merge
// (record mode: per-warp partials of every (sequence, KV head) unit) and the chunk merge
// (chunk-merge mode: per-CTA partials of every query row).
//
// A record r holds, for each of the unit's (at most 4) query heads h, the warp's running
// maximum m_rh of the base-2 logits, its sum l_rh = sum 2^(s - m_rh) and the unnormalized
// O_rh = sum 2^(s - m_rh) v (register order of the decode kernel's accumulators).  The
// output is the flash-decode reduction of the split over kv_len:
//   M_h = max_r m_rh,  out_h = sum_r 2^(m_rh - M_h) O_rh / sum_r 2^(m_rh - M_h) l_rh.
// Records with m = -inf (warps or CTAs that saw no token) contribute nothing.  Every sum
// runs in a fixed order, so the result does not depend on the order in which the decode
// kernel's warps finished.
//
// Grid: (slices of a record, units).  A CTA's 512 threads are NQ float4 positions x
// 512 / NQ record groups, NQ chosen from the records per unit: 8 positions x 64 groups for
// many records (a record in 16 or 8 slices), up to a whole record per CTA x 4 groups for a
// few, so that the grid does not grow past what the records need (with 512 units of 4
// records, 16 CTAs per unit of mostly idle groups ran for ~100 us).  Each thread loads the O values
// of its records first (one round trip for up to 8 per group), the CTA meanwhile forms the
// per-head maxima, weights and denominators from all records' (m, l), and the weighted
// sums meet in shared memory.
// Launched with programmatic stream serialization right after the decode kernel: its CTAs
// start as the decode's CTAs leave and wait (griddepcontrol.wait) for that grid's writes.
#include "kvq_decode_mma.cuh"

namespace kvq {

namespace {

constexpr int kMergeThreads = 512;
constexpr int kBatch = 8;                     // records per thread per round of loads

__device__ __forceinline__ float4 ld_cg4(const float4* p) { return __ldcg(p); }

// Block-wide max / sum of four values (fixed tree: lanes, then warps in order).
__device__ __forceinline__ void block_reduce4(float* v, bool is_max, float (*red)[4], float* res) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float o = __shfl_xor_sync(0xffffffffu, v[h], off);
      v[h] = is_max ? fmaxf(v[h], o) : v[h] + o;
    }
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < 4; ++h) red[warp][h] = v[h];
  __syncthreads();
  if (threadIdx.x < 4) {
    float r = red[0][threadIdx.x];
    for (int w = 1; w < kMergeThreads / 32; ++w) r = is_max ? fmaxf(r, red[w][threadIdx.x]) : r + red[w][threadIdx.x];
    res[threadIdx.x] = r;
  }
  __syncthreads();
}

template <int VC, int D, int kNQ>
__global__ void __launch_bounds__(kMergeThreads, 2) record_merge_kernel(DecodeArgs a) {
  constexpr int P = D / 16 * 64;              // floats per record (4 heads x D)
  constexpr int kNG = kMergeThreads / kNQ;    // record groups
  static_assert(kNQ * 4 <= P && kNG >= 4, "slice shape");
  // partial sums meet per warp (groups of a warp summed by shuffles first) for NQ < 32,
  // per group otherwise
  constexpr int kRG = kNQ < 32 ? kMergeThreads / 32 : kNG;
  extern __shared__ float w_sm[];             // [R][4] weights 2^(m - M)
  __shared__ float red[kMergeThreads / 32][4];
  __shared__ float sM[4], sden[4];
  __shared__ float4 racc[kRG][kNQ];
  const int tid = threadIdx.x, q = tid & (kNQ - 1), g = tid / kNQ;
  const int R = a.warp_records;
  const long long unit = blockIdx.y;
  const int slice = blockIdx.x;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (a.seq_lens_adv && slice == 0 && unit % a.k.num_kv_heads == 0 && tid == 0) {
    // fused step: every CTA of the decode grid has read seq_lens[b] (that grid is complete),
    // so the new length is stored here, under the decode kernel's own length check
    const long long b = unit / a.k.num_kv_heads;
    const long long cap = min((long long)a.max_pages * a.k.page_size, (long long)a.n_chunks * a.chunk_tokens);
    const long long L_old = a.seq_lens_adv[b];
    if (L_old >= 0 && L_old + 1 <= cap) a.seq_lens_adv[b] = (int32_t)(L_old + 1);
  }

  const float4* ml4 = reinterpret_cast<const float4*>(a.part_ml + unit * R * 8);
  const float4* po = reinterpret_cast<const float4*>(a.part_o + unit * R * P) + slice * kNQ + q;
  // this thread's first batch of O values, in flight while the weights are formed
  float4 ov[kBatch];
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int r = g + u * kNG;
    if (r < R) ov[u] = ld_cg4(po + (long long)r * (P / 4));
  }
  // per-head maxima over the records
  float v[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
  for (int r = tid; r < R; r += kMergeThreads) {
    const float4 x = ld_cg4(ml4 + 2 * r), y = ld_cg4(ml4 + 2 * r + 1);
    v[0] = fmaxf(v[0], x.x); v[1] = fmaxf(v[1], x.z); v[2] = fmaxf(v[2], y.x); v[3] = fmaxf(v[3], y.z);
  }
  block_reduce4(v, true, red, sM);
  // weights and denominators
  float M[4], den[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
  for (int h = 0; h < 4; ++h) M[h] = sM[h];
  for (int r = tid; r < R; r += kMergeThreads) {
    const float4 x = ld_cg4(ml4 + 2 * r), y = ld_cg4(ml4 + 2 * r + 1);
    const float m[4] = {x.x, x.z, y.x, y.z}, l[4] = {x.y, x.w, y.y, y.w};
    float4 w;
    float* wp = &w.x;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      wp[h] = m[h] == -INFINITY ? 0.0f : fast_exp2(m[h] - M[h]);
      den[h] = fmaf(wp[h], l[h], den[h]);
    }
    reinterpret_cast<float4*>(w_sm)[r] = w;
  }
  block_reduce4(den, false, red, sden);   // its barriers also publish w_sm

  // weighted sum of this thread's records; the components of a float4 position are heads
  // 0, 1, 2, 3 (positions 4j .. 4j + 3: lanes 2j, 2j + 1 of the accumulator layout, k = 0, 1)
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  auto fold = [&](int r, const float4& o) {
    const float4 w = reinterpret_cast<const float4*>(w_sm)[r];
    if (w.x != 0.0f) acc.x = fmaf(w.x, o.x, acc.x);
    if (w.y != 0.0f) acc.y = fmaf(w.y, o.y, acc.y);
    if (w.z != 0.0f) acc.z = fmaf(w.z, o.z, acc.z);
    if (w.w != 0.0f) acc.w = fmaf(w.w, o.w, acc.w);
  };
#pragma unroll
  for (int u = 0; u < kBatch; ++u) {
    const int r = g + u * kNG;
    if (r < R) fold(r, ov[u]);
  }
  for (int r0 = g + kBatch * kNG; r0 < R; r0 += kBatch * kNG) {   // more than 512 records
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int r = r0 + u * kNG;
      if (r < R) ov[u] = ld_cg4(po + (long long)r * (P / 4));
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int r = r0 + u * kNG;
      if (r < R) fold(r, ov[u]);
    }
  }
  // over the record groups: lanes of a warp with the same q (NQ < 32: the groups of a
  // warp), then warps or groups, in a fixed order
  if constexpr (kNQ < 32) {
#pragma unroll
    for (int off = kNQ; off < 32; off <<= 1) {
      acc.x += __shfl_xor_sync(0xffffffffu, acc.x, off);
      acc.y += __shfl_xor_sync(0xffffffffu, acc.y, off);
      acc.z += __shfl_xor_sync(0xffffffffu, acc.z, off);
      acc.w += __shfl_xor_sync(0xffffffffu, acc.w, off);
    }
    if ((tid & 31) < kNQ) racc[tid >> 5][q] = acc;
  } else {
    racc[g][q] = acc;
  }
  __syncthreads();
  for (int t4 = tid; t4 < kNQ * 4; t4 += kMergeThreads) {
    const int qq = t4 >> 2, c = t4 & 3;
    float sum = 0.0f;
    for (int w = 0; w < kRG; ++w) sum += (&racc[w][qq].x)[c];
    const int t = slice * kNQ * 4 + qq * 4 + c;      // position in the record
    const int mt = t >> 6, ln = (t >> 1) & 31, rr = ln >> 2, ii = ln & 3;
    const int dim = mma::pv_dim<VC>(mt, ii < 2 ? rr : rr + 8);
    const int h = 2 * (ii & 1) + (t & 1);
    const int G = a.group, gcount = G < 4 ? G : 4;
    if (h < gcount) {
      const long long kvh = unit % a.k.num_kv_heads, b = unit / a.k.num_kv_heads;
      const long long head = b * a.num_q_heads + kvh * G + h;
      const float d = sden[h];
      a.out[head * D + dim] = d > 0.0f ? __fdividef(sum, d) : 0.0f;
    }
  }
}

template <int VC, int D, int kNQ>
cudaError_t launch_merge_nq(const DecodeArgs& a, cudaStream_t stream) {
  auto kern = record_merge_kernel<VC, D, kNQ>;
  const size_t smem = (size_t)a.warp_records * 16;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  constexpr int P = D / 16 * 64;
  const dim3 grid(P / (kNQ * 4), (unsigned)(a.batch * a.k.num_kv_heads));
  const cudaError_t e = launch_pdl(kern, grid, dim3(kMergeThreads), smem, stream, a);
  count_launch();
  return e;
}

// Slice shape from the records per unit: about one round of loads per group (8 records)
// while that keeps 4 or more groups per CTA.
template <int VC, int D>
cudaError_t launch_merge(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int P4 = D / 16 * 16;   // float4 positions per record
  const int R = a.warp_records;
  if (R <= 4 * kBatch) return launch_merge_nq<VC, D, P4>(a, stream);                    // 512 / P4 groups
  if (R <= 16 * kBatch) return launch_merge_nq<VC, D, 32>(a, stream);                   // 16 groups
  return launch_merge_nq<VC, D, 8>(a, stream);                                          // 64 groups
}

template <int VC>
cudaError_t launch_merge_d(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  if (head_dim == 64) return launch_merge<VC, 64>(a, stream);
  if (head_dim == 128) return launch_merge<VC, 128>(a, stream);
  return cudaErrorNotSupported;
}

// ---------------------------------------------------------------- chunk merge
// Split-K combine (step a8) for the chunk-merge mode of the heads-on-M loop: merges the
// n_chunks chunk partials (m_c, l_c, O_c) of every query row into its output,
//   M = max_c m_c,  out = sum_c 2^(m_c - M) O_c / sum_c 2^(m_c - M) l_c,
// skipping partials with m = -inf (chunks without tokens; their O is not written).
// Grid: (slices of head_dim, query rows).  256 threads = COLS float4 columns x 256 / COLS
// chunk groups (a whole row for few chunks, 64-element slices x 16 groups for many); each
// thread loads the O values of its chunks (c = group, group + groups, ...) first, the CTA
// forms the weights from all chunks' (m, l) meanwhile, and the groups' sums meet in shared
// memory in a fixed order.
constexpr int kCmThreads = 256, kCmBatch = 8;

__device__ __forceinline__ float block_reduce1(float v, bool is_max, float* red, float* res) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(0xffffffffu, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    float r = red[0];
    for (int w = 1; w < kCmThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    *res = r;
  }
  __syncthreads();
  return *res;
}

template <int D, int kCmCols>
__global__ void __launch_bounds__(kCmThreads) chunk_merge_kernel(DecodeArgs a) {
  constexpr int kCmGroups = kCmThreads / kCmCols;   // chunk groups
  extern __shared__ float cw[];                 // [n_chunks] weights 2^(m_c - M)
  __shared__ float red[kCmThreads / 32];
  __shared__ float sres[2];
  __shared__ float4 racc[kCmGroups][kCmCols];
  const int tid = threadIdx.x, q = tid % kCmCols, g = tid / kCmCols;
  const int n = a.n_chunks;
  const long long row = blockIdx.y;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const float2* ml = reinterpret_cast<const float2*>(a.part_ml) + row * n;
  const float4* po = reinterpret_cast<const float4*>(a.part_o + row * n * D) + blockIdx.x * kCmCols + q;
  // this thread's first batch of O values, in flight while the weights are formed
  float4 ov[kCmBatch];
#pragma unroll
  for (int u = 0; u < kCmBatch; ++u) {
    const int c = g + u * kCmGroups;
    if (c < n) ov[u] = __ldcg(po + (long long)c * (D / 4));
  }
  float m = -INFINITY;
  for (int c = tid; c < n; c += kCmThreads) m = fmaxf(m, __ldcg(ml + c).x);
  const float M = block_reduce1(m, true, red, &sres[0]);
  float den = 0.0f;
  for (int c = tid; c < n; c += kCmThreads) {
    const float2 x = __ldcg(ml + c);
    const float w = x.x == -INFINITY ? 0.0f : fast_exp2(x.x - M);
    cw[c] = w;
    den = fmaf(w, x.y, den);
  }
  den = block_reduce1(den, false, red, &sres[1]);   // its barriers also publish cw
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  auto fold = [&](int c, const float4& o) {
    const float w = cw[c];
    if (w != 0.0f) {
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
  };
#pragma unroll
  for (int u = 0; u < kCmBatch; ++u) {
    const int c = g + u * kCmGroups;
    if (c < n) fold(c, ov[u]);
  }
  for (int c0 = g + kCmBatch * kCmGroups; c0 < n; c0 += kCmBatch * kCmGroups) {
#pragma unroll
    for (int u = 0; u < kCmBatch; ++u) {
      const int c = c0 + u * kCmGroups;
      if (c < n) ov[u] = __ldcg(po + (long long)c * (D / 4));
    }
#pragma unroll
    for (int u = 0; u < kCmBatch; ++u) {
      const int c = c0 + u * kCmGroups;
      if (c < n) fold(c, ov[u]);
    }
  }
  racc[g][q] = acc;
  __syncthreads();
  if (tid < kCmCols) {
    float4 sum = racc[0][tid];
    for (int gg = 1; gg < kCmGroups; ++gg) {
      const float4 x = racc[gg][tid];
      sum.x += x.x; sum.y += x.y; sum.z += x.z; sum.w += x.w;
    }
    const float inv = den > 0.0f ? 1.0f / den : 0.0f;
    reinterpret_cast<float4*>(a.out + row * D)[blockIdx.x * kCmCols + tid] =
        make_float4(sum.x * inv, sum.y * inv, sum.z * inv, sum.w * inv);
  }
}

template <int D, int kCmCols>
cudaError_t launch_cm_cols(const DecodeArgs& a, cudaStream_t stream) {
  auto kern = chunk_merge_kernel<D, kCmCols>;
  const size_t smem = (size_t)a.n_chunks * 4;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  const dim3 grid(D / (4 * kCmCols), (unsigned)((long long)a.batch * a.num_q_heads));
  const cudaError_t e = launch_pdl(kern, grid, dim3(kCmThreads), smem, stream, a);
  count_launch();
  return e;
}

// Slice shape from the chunks per row: a whole row per CTA while its groups take every
// chunk in one round of loads (a batch of many rows and few chunks then runs as many CTAs
// as rows instead of D / 64 times as many), else 64-element slices with 16 chunk groups.
template <int D>
cudaError_t launch_cm(const DecodeArgs& a, cudaStream_t stream) {
  constexpr int kRowCols = D / 4;                      // float4 columns of a row
  if (a.n_chunks <= (kCmThreads / kRowCols) * kCmBatch) return launch_cm_cols<D, kRowCols>(a, stream);
  return launch_cm_cols<D, 16>(a, stream);
}

}  // namespace

cudaError_t launch_chunk_merge_pdl(const DecodeArgs& a, int head_dim, cudaStream_t stream) {
  if (head_dim == 128) return launch_cm<128>(a, stream);
  if (head_dim == 256) return launch_cm<256>(a, stream);
  return cudaErrorNotSupported;
}

cudaError_t launch_record_merge_pdl(const DecodeArgs& a, int head_dim, int v_codec, cudaStream_t stream) {
  switch (v_codec) {
    case KVQ_CODEC_Q8_0: return launch_merge_d<KVQ_CODEC_Q8_0>(a, head_dim, stream);
    case KVQ_CODEC_Q4S: return launch_merge_d<KVQ_CODEC_Q4S>(a, head_dim, stream);
    case KVQ_CODEC_BF16: return launch_merge_d<KVQ_CODEC_BF16>(a, head_dim, stream);
    case KVQ_CODEC_F16: return launch_merge_d<KVQ_CODEC_F16>(a, head_dim, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace kvq
