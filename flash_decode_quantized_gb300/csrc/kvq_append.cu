// On-device encode of new K/V rows into the resident paged store (step a1).
//
// rMLX issue #295 ("Root cause", "Fix direction") traces the K-only codecs' gap to the
// growing prefix being restaged through the host on every step and asks for the
// prefix to stay resident so the kernel reads the quant store directly; this kernel is
// the on-device half of that: each new row is quantized where it will be read.
//
// One warp encodes one row (one token of one KV head) with encode_row.

#include <climits>

#include "kvq_encode.cuh"
#include "kvq_internal.cuh"

namespace kvq {

namespace {

constexpr int kWarpsPerBlock = 8;

template <int CODEC, int EPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
append_kernel(StoreView st, const __nv_bfloat16* __restrict__ rows, int n_new, int batch,
              const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ page_table,
              int max_pages) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long row_id = (long long)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
  const long long n_rows = (long long)batch * n_new * st.num_kv_heads;
  if (row_id >= n_rows) return;
  const int h = (int)(row_id % st.num_kv_heads);
  const long long bi = row_id / st.num_kv_heads;
  const int i = (int)(bi % n_new);
  const int b = (int)(bi / n_new);
  encode_row<CODEC, EPL>(st, rows, row_id, n_new, (long long)seq_lens[b], b, i, h, page_table, max_pages);
}

// K and V rows of one step in one launch.  CTA (x, b) encodes warps' worth of sequence
// b's rows: the first n_new*Hkv row slots are K rows, the next n_new*Hkv are V rows.
// With `advance` (only when one CTA covers a sequence), the CTA adds n_new to
// seq_lens[b] after every warp has read it.
template <int KCODEC, int VCODEC, int EPL>
__global__ void __launch_bounds__(512)
append_kv_kernel(StoreView ks, StoreView vs, const __nv_bfloat16* __restrict__ k_rows,
                 const __nv_bfloat16* __restrict__ v_rows, int n_new, int32_t* __restrict__ seq_lens,
                 const int32_t* __restrict__ page_table, int max_pages, int advance) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.y;
  const long long per_store = (long long)n_new * ks.num_kv_heads;
  const long long slot = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const long long base = seq_lens[b];
  if (slot < 2 * per_store) {
    const bool is_v = slot >= per_store;
    const long long r = is_v ? slot - per_store : slot;   // row within this sequence
    const int h = (int)(r % ks.num_kv_heads);
    const int i = (int)(r / ks.num_kv_heads);
    const long long row_id = (long long)b * per_store + r;
    if (is_v) encode_row<VCODEC, EPL>(vs, v_rows, row_id, n_new, base, b, i, h, page_table, max_pages);
    else encode_row<KCODEC, EPL>(ks, k_rows, row_id, n_new, base, b, i, h, page_table, max_pages);
  }
  if (advance) {
    __syncthreads();
    if (threadIdx.x == 0) seq_lens[b] = (int32_t)(base + n_new);
  }
}

// Bulk encode (prompt-sized appends).  A CTA takes kBulkPos consecutive new positions of
// one sequence and encodes their rows for every KV head (for both stores with TWO).
constexpr int kBulkPos = 16;
constexpr int kBulkRows = 4;
constexpr int kBulkThreads = 256;

template <int KC, int VC, int EPL, bool TWO>
__global__ void __launch_bounds__(kBulkThreads)
append_bulk_kernel(StoreView ks, StoreView vs, const __nv_bfloat16* __restrict__ k_rows,
                   const __nv_bfloat16* __restrict__ v_rows, int n_new, const int32_t* __restrict__ seq_lens,
                   const int32_t* __restrict__ page_table, int max_pages) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int D = EPL * 32;
  constexpr int NW = kBulkThreads / 32;
  const int b = blockIdx.y, i0 = blockIdx.x * kBulkPos;
  const int H = ks.num_kv_heads;
  const int P = ks.page_size;
  const int npos = min(kBulkPos, n_new - i0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long base = seq_lens[b];
  const long long cap = min((long long)max_pages * P, (long long)INT_MAX);
  // one warp per position: its page is looked up once, then every KV head's K and V rows
  // are encoded, kBulkRows rows' loads in flight at a time (no integer divisions per row)
  for (int ip = warp; ip < npos; ip += NW) {
    const int i = i0 + ip;
    const long long pos_ll = base + i;
    if (base < 0 || pos_ll >= cap) {
      if (lane == 0) {
        record_fault(ks.status, KVQ_DEVICE_BAD_POSITION);
        if (TWO) record_fault(vs.status, KVQ_DEVICE_BAD_POSITION);
      }
      continue;
    }
    const int pos = (int)pos_ll;
    const int page = page_table[(long long)b * max_pages + pos / P];
    const int r = pos % P;
    const long long row0 = ((long long)b * n_new + i) * H;   // row of head 0 of this position
#pragma unroll
    for (int which = 0; which < (TWO ? 2 : 1); ++which) {
      const StoreView& st = which ? vs : ks;
      if (page < 0 || page >= st.num_pages) {
        if (lane == 0) record_fault(st.status, KVQ_DEVICE_BAD_PAGE);
        continue;
      }
      const __nv_bfloat16* src = (which ? v_rows : k_rows) + row0 * D;
      for (int h0 = 0; h0 < H; h0 += kBulkRows) {
        float x[kBulkRows][EPL];
#pragma unroll
        for (int u = 0; u < kBulkRows; ++u)
          if (h0 + u < H) load_row<EPL>(src + (long long)(h0 + u) * D, lane, x[u]);
#pragma unroll
        for (int u = 0; u < kBulkRows; ++u) {
          if (h0 + u >= H) break;
          if (which) store_row<VC, EPL>(vs, page, r, h0 + u, x[u]);
          else store_row<KC, EPL>(ks, page, r, h0 + u, x[u]);
        }
      }
    }
  }
}

template <int KC, int VC, bool TWO>
cudaError_t launch_bulk(const kvq_store* ks, const kvq_store* vs, const __nv_bfloat16* k_rows,
                        const __nv_bfloat16* v_rows, int n_new, int batch, const int32_t* seq_lens,
                        const int32_t* page_table, int max_pages, cudaStream_t stream) {
  const dim3 grid((unsigned)((n_new + kBulkPos - 1) / kBulkPos), batch);
  const StoreView kv = view_of(ks), vv = view_of(TWO ? vs : ks);
  cudaError_t e;
  switch (ks->desc.head_dim) {
    case 64: e = launch_pdl(append_bulk_kernel<KC, VC, 2, TWO>, grid, dim3(kBulkThreads), 0, stream, kv, vv, k_rows, v_rows, n_new, seq_lens, page_table, max_pages); break;
    case 128: e = launch_pdl(append_bulk_kernel<KC, VC, 4, TWO>, grid, dim3(kBulkThreads), 0, stream, kv, vv, k_rows, v_rows, n_new, seq_lens, page_table, max_pages); break;
    case 256: e = launch_pdl(append_bulk_kernel<KC, VC, 8, TWO>, grid, dim3(kBulkThreads), 0, stream, kv, vv, k_rows, v_rows, n_new, seq_lens, page_table, max_pages); break;
    default: return cudaErrorNotSupported;
  }
  count_launch();
  return e;
}

template <int CODEC>
cudaError_t launch_codec(const kvq_store* s, const __nv_bfloat16* rows, int n_new, int batch,
                         const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                         cudaStream_t stream) {
  if (n_new >= kBulkPos)   // prompt-sized: rows of a sequence's positions per CTA
    return launch_bulk<CODEC, CODEC, false>(s, s, rows, rows, n_new, batch, seq_lens, page_table, max_pages, stream);
  const long long n_rows = (long long)batch * n_new * s->desc.num_kv_heads;
  const unsigned grid = (unsigned)((n_rows + kWarpsPerBlock - 1) / kWarpsPerBlock);
  const StoreView v = view_of(s);
  // same carveout as the decode kernels, so a step's kernels run without reconfiguring
  static bool carveout_set = false;
  if (!carveout_set) {
    cudaFuncSetAttribute(append_kernel<CODEC, 2>, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    cudaFuncSetAttribute(append_kernel<CODEC, 4>, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    cudaFuncSetAttribute(append_kernel<CODEC, 8>, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    carveout_set = true;
  }
  cudaError_t e;
  switch (s->desc.head_dim) {
    case 64:
      e = launch_pdl(append_kernel<CODEC, 2>, dim3(grid), dim3(kWarpsPerBlock * 32), 0, stream, v, rows, n_new, batch, seq_lens, page_table, max_pages);
      break;
    case 128:
      e = launch_pdl(append_kernel<CODEC, 4>, dim3(grid), dim3(kWarpsPerBlock * 32), 0, stream, v, rows, n_new, batch, seq_lens, page_table, max_pages);
      break;
    case 256:
      e = launch_pdl(append_kernel<CODEC, 8>, dim3(grid), dim3(kWarpsPerBlock * 32), 0, stream, v, rows, n_new, batch, seq_lens, page_table, max_pages);
      break;
    default:
      return cudaErrorNotSupported;
  }
  count_launch();
  return e;
}

__global__ void seq_lens_add_kernel(int32_t* seq_lens, int batch, int n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < batch) seq_lens[b] += n;
}

template <int KC, int VC>
cudaError_t launch_kv_pair(const kvq_store* ks, const kvq_store* vs, const __nv_bfloat16* k_rows,
                           const __nv_bfloat16* v_rows, int n_new, int batch, int32_t* seq_lens,
                           const int32_t* page_table, int max_pages, int advance, cudaStream_t stream) {
  if (n_new >= kBulkPos) {   // prompt-sized: the bulk kernel, then the advance
    cudaError_t e = launch_bulk<KC, VC, true>(ks, vs, k_rows, v_rows, n_new, batch, seq_lens, page_table,
                                              max_pages, stream);
    if (e != cudaSuccess || !advance) return e;
    return launch_seq_lens_add(seq_lens, batch, n_new, stream);
  }
  const long long slots = 2LL * n_new * ks->desc.num_kv_heads;   // warps per sequence
  const int warps = (int)(slots < 16 ? slots : 16);
  const unsigned gx = (unsigned)((slots + warps - 1) / warps);
  const int adv = (advance && gx == 1) ? 1 : 0;
  const StoreView kv = view_of(ks), vv = view_of(vs);
  cudaError_t e;
  switch (ks->desc.head_dim) {
    case 64: e = launch_pdl(append_kv_kernel<KC, VC, 2>, dim3(gx, batch), dim3(32 * warps), 0, stream, kv, vv, k_rows, v_rows, n_new, seq_lens, page_table, max_pages, adv); break;
    case 128: e = launch_pdl(append_kv_kernel<KC, VC, 4>, dim3(gx, batch), dim3(32 * warps), 0, stream, kv, vv, k_rows, v_rows, n_new, seq_lens, page_table, max_pages, adv); break;
    case 256: e = launch_pdl(append_kv_kernel<KC, VC, 8>, dim3(gx, batch), dim3(32 * warps), 0, stream, kv, vv, k_rows, v_rows, n_new, seq_lens, page_table, max_pages, adv); break;
    default: return cudaErrorNotSupported;
  }
  count_launch();
  if (e != cudaSuccess || !advance || adv) return e;
  // several CTAs per sequence: advance in a separate launch, after all of them
  return launch_seq_lens_add(seq_lens, batch, n_new, stream);
}

template <int KC>
cudaError_t launch_kv_v(const kvq_store* ks, const kvq_store* vs, const __nv_bfloat16* k_rows,
                        const __nv_bfloat16* v_rows, int n_new, int batch, int32_t* seq_lens,
                        const int32_t* page_table, int max_pages, int advance, cudaStream_t stream) {
  switch (vs->desc.codec) {
    case KVQ_CODEC_BF16: return launch_kv_pair<KC, KVQ_CODEC_BF16>(ks, vs, k_rows, v_rows, n_new, batch, seq_lens, page_table, max_pages, advance, stream);
    case KVQ_CODEC_F16: return launch_kv_pair<KC, KVQ_CODEC_F16>(ks, vs, k_rows, v_rows, n_new, batch, seq_lens, page_table, max_pages, advance, stream);
    case KVQ_CODEC_Q8_0: return launch_kv_pair<KC, KVQ_CODEC_Q8_0>(ks, vs, k_rows, v_rows, n_new, batch, seq_lens, page_table, max_pages, advance, stream);
    case KVQ_CODEC_Q4S: return launch_kv_pair<KC, KVQ_CODEC_Q4S>(ks, vs, k_rows, v_rows, n_new, batch, seq_lens, page_table, max_pages, advance, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace

cudaError_t launch_append(const kvq_store* s, const __nv_bfloat16* rows, int n_new, int batch,
                          const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                          cudaStream_t stream) {
  switch (s->desc.codec) {
    case KVQ_CODEC_BF16: return launch_codec<KVQ_CODEC_BF16>(s, rows, n_new, batch, seq_lens, page_table, max_pages, stream);
    case KVQ_CODEC_F16: return launch_codec<KVQ_CODEC_F16>(s, rows, n_new, batch, seq_lens, page_table, max_pages, stream);
    case KVQ_CODEC_Q8_0: return launch_codec<KVQ_CODEC_Q8_0>(s, rows, n_new, batch, seq_lens, page_table, max_pages, stream);
    case KVQ_CODEC_Q4S: return launch_codec<KVQ_CODEC_Q4S>(s, rows, n_new, batch, seq_lens, page_table, max_pages, stream);
    default: return cudaErrorNotSupported;
  }
}

cudaError_t launch_seq_lens_add(int32_t* seq_lens, int batch, int n, cudaStream_t stream) {
  const cudaError_t e = launch_pdl(seq_lens_add_kernel, dim3((batch + 255) / 256), dim3(256), 0, stream, seq_lens, batch, n);
  count_launch();
  return e;
}

cudaError_t launch_append_kv(const kvq_store* ks, const kvq_store* vs, const __nv_bfloat16* k_rows,
                             const __nv_bfloat16* v_rows, int n_new, int batch, int32_t* seq_lens,
                             const int32_t* page_table, int max_pages, int advance, cudaStream_t stream) {
  switch (ks->desc.codec) {
    case KVQ_CODEC_BF16: return launch_kv_v<KVQ_CODEC_BF16>(ks, vs, k_rows, v_rows, n_new, batch, seq_lens, page_table, max_pages, advance, stream);
    case KVQ_CODEC_F16: return launch_kv_v<KVQ_CODEC_F16>(ks, vs, k_rows, v_rows, n_new, batch, seq_lens, page_table, max_pages, advance, stream);
    case KVQ_CODEC_Q8_0: return launch_kv_v<KVQ_CODEC_Q8_0>(ks, vs, k_rows, v_rows, n_new, batch, seq_lens, page_table, max_pages, advance, stream);
    case KVQ_CODEC_Q4S: return launch_kv_v<KVQ_CODEC_Q4S>(ks, vs, k_rows, v_rows, n_new, batch, seq_lens, page_table, max_pages, advance, stream);
    default: return cudaErrorNotSupported;
  }
}

}  // namespace kvq
