// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvq.h"

struct kvq_store {
  CUtensorMap rows_map;  // TMA map of the row data: {row_bytes, page_size, kv_heads, pages}
  bool rows_map_ok;
  kvq_store_desc desc;
  uint8_t* buf;        // caller-owned device memory
  size_t bytes;
  int32_t* status;     // device status word, owned by the handle
  int device;
  int row_bytes;       // bytes of one row's data
  int n_scales;        // fp16 scales per row (0 for 16-bit codecs)
  long long slab_bytes;  // one (page, head) slab
};

namespace kvq {

constexpr int kBlock = 32;       // elements per quantization block
constexpr int kMergeGroup = 16;  // split-K chunks merged per group partial

__host__ __device__ inline int codec_row_bytes(int codec, int head_dim) {
  return codec == KVQ_CODEC_Q8_0 ? head_dim : codec == KVQ_CODEC_Q4S ? head_dim / 2 : 2 * head_dim;
}
__host__ __device__ inline int codec_scales(int codec, int head_dim) {
  return (codec == KVQ_CODEC_Q8_0 || codec == KVQ_CODEC_Q4S) ? head_dim / kBlock : 0;
}

// Records the first device fault in a status word (first writer wins, never traps).
__device__ inline void record_fault(int32_t* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// Geometry of one store as the kernels see it.
struct StoreView {
  const uint8_t* buf;
  int32_t* status;
  long long slab_bytes;
  int row_bytes;
  int n_scales;
  int num_pages;
  int num_kv_heads;
  int page_size;
};

inline StoreView view_of(const kvq_store* s) {
  StoreView v;
  v.buf = s->buf;
  v.status = s->status;
  v.slab_bytes = s->slab_bytes;
  v.row_bytes = s->row_bytes;
  v.n_scales = s->n_scales;
  v.num_pages = s->desc.num_pages;
  v.num_kv_heads = s->desc.num_kv_heads;
  v.page_size = s->desc.page_size;
  return v;
}

// Arguments common to the decode kernels.
struct DecodeArgs {
  const __nv_bfloat16* q;      // [B][Hq][D]
  StoreView k, v;
  const int32_t* seq_lens;     // [B]
  const int32_t* page_table;   // [B][max_pages]
  int max_pages;
  int batch;
  int num_q_heads;             // query rows per sequence: Hq * tokens
  int group;                   // query rows per KV head: (Hq / Hkv) * tokens
  int tokens;                  // query tokens per sequence; q/out are [B][Hq][tokens][D] and
                               // query token i attends to positions < seq_len - tokens + 1 + i
  float qk_scale_log2;         // softmax scale * log2(e)
  int chunk_tokens;            // split-K chunk length
  int n_chunks;                // chunks per (sequence, kv head)
  float* part_o;               // [B][Hq][n_chunks][D]
  float* part_ml;              // [B][Hq][n_chunks][2]  (running max in log2 units, sum)
  float* gpart_o;              // [B][Hq][n_groups][D]  group partials of the split
  float* gpart_ml;             // [B][Hq][n_groups][2]
  int n_groups;                // groups of chunks per (sequence, kv head)
  unsigned* counters;          // [B*Hkv] unit counters, then [B*Hkv][n_groups] group
                               // counters at grp_counter_off (all zero between calls)
  long long grp_counter_off;
  float* out;                  // [B][Hq][D]
  // Fused append (tensor-core kernel only): with k_new set, the token at position
  // seq_lens[b] gets rows k_new/v_new [B][Hkv][D] (bf16) written by the CTA whose tile
  // holds it, and attention covers seq_lens[b] + 1 tokens.  With seq_lens_adv set as
  // well, the last of the sequence's CTAs to have read seq_lens[b] (counted in
  // seq_counters[b], zero between calls) stores seq_lens[b] + 1 there.
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int32_t* seq_lens_adv;
  unsigned* seq_counters;
  // Record mode (warps of at most 4 heads, D <= 128): with warp_records > 0 the decode
  // kernel merges nothing; every warp writes its own partial as record
  // (chunk * pipes + pipe) * 4 + slice of its (sequence, KV head) unit:
  //   part_ml [unit][record][8]: (m, l) of heads 0, 1, 2, 3 (base-2 max, sum)
  //   part_o  [unit][record][D * 4]: unnormalized O in the accumulator's register order
  // and the record merge kernel (launched right after it) forms the output.
  int warp_records;
  // Chunk-merge mode (heads-on-M loop): every CTA writes its chunk partial (m = -inf for a
  // CTA without tokens) to part_ml / part_o and the chunk merge kernel, launched right
  // after it, combines them into the output (no arrival counters, no in-place merge).
  int chunk_merge;
  int solo;                    // at most 4 query rows per KV head: one pipeline per CTA (Cfg SOLO)
  int wait_limit;              // tries of each bounded mbarrier wait before it gives up
  int skip_tile;               // fault injection: tile the first pipeline never issues (-1: none)
};

// Arguments of the prefill attention kernel (kvq_prefill.cuh).
struct PrefillArgs {
  const __nv_bfloat16* q;     // [B][T][Hq][D]
  StoreView k, v;
  const int32_t* seq_lens;    // [B], counting the T new tokens
  const int32_t* page_table;  // [B][max_pages]
  int max_pages;
  int num_q_heads;
  int group;                  // Hq / Hkv
  int tokens;                 // T
  float qk_scale_log2;
  float* out;                 // [B][T][Hq][D]
  int wait_limit;             // tries of each bounded mbarrier wait (tensor-core kernel)
  int skip_tile;              // fault injection: tile the producer never issues (-1: none)
};

// Launchers implemented in the kernel translation units.  Each returns a CUDA error.
cudaError_t launch_append(const kvq_store* store, const __nv_bfloat16* rows, int n_new, int batch,
                          const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                          cudaStream_t stream);
cudaError_t launch_seq_lens_add(int32_t* seq_lens, int batch, int n, cudaStream_t stream);
cudaError_t launch_dequantize(const kvq_store* src, kvq_store* dst, const int32_t* seq_lens,
                              const int32_t* page_table, int max_pages, int batch, cudaStream_t stream);
cudaError_t launch_append_kv(const kvq_store* ks, const kvq_store* vs, const __nv_bfloat16* k_rows,
                             const __nv_bfloat16* v_rows, int n_new, int batch, int32_t* seq_lens,
                             const int32_t* page_table, int max_pages, int advance, cudaStream_t stream);

// Launches `kern` with programmatic stream serialization: the launch may begin while the
// stream's previous kernel finishes; every kernel of this library waits on
// griddepcontrol.wait before touching data a previous kernel may write.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
cudaError_t launch_combine_pdl(const DecodeArgs& a, int head_dim, cudaStream_t stream);
cudaError_t launch_chunk_merge_pdl(const DecodeArgs& a, int head_dim, cudaStream_t stream);
cudaError_t launch_record_merge_pdl(const DecodeArgs& a, int head_dim, int v_codec, cudaStream_t stream);

void count_launch();
// Fault injection for tests of the timeout path (kvq_set_fault_injection): the wait limit
// and the skipped tile that the next decode launches use.
void fault_injection(int* wait_limit, int* skip_tile);
kvq_status decode_workspace_layout(const kvq_store* k_store, const kvq_store* v_store, int batch,
                                   int num_q_heads, int max_len_hint, const kvq_decode_opts* opts,
                                   size_t* total, size_t* counters_off);
// kvq_flash_decode that zeroes the workspace's counters on the stream right before its
// launch, once every argument check has passed (nothing is enqueued on a failed check).
kvq_status decode_reset(const void* q, const kvq_store* k_store, const kvq_store* v_store,
                        const int32_t* seq_lens, const int32_t* page_table, int max_pages, kvq_codec codec,
                        float* out, int batch, int num_q_heads, float softmax_scale, int max_len_hint,
                        const kvq_decode_opts* opts, void* workspace, size_t workspace_bytes, void* stream);

}  // namespace kvq
