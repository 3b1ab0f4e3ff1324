// Host side of the C ABI declared in include/kvq.h: argument checks, store handles, the
// split planner and the kernel launches.  No call here waits for the device except
// kvq_store_get_error, and none copies data to or from the host.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdlib>
#include <mutex>
#include <new>

#include "kvq_internal.cuh"

namespace kvq {

static std::atomic<unsigned long long> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

static std::atomic<int> g_wait_limit{0};   // 0: the default limit
static std::atomic<int> g_skip_tile{-1};
void fault_injection(int* wait_limit, int* skip_tile) {
  const int w = g_wait_limit.load(std::memory_order_relaxed);
  *wait_limit = w > 0 ? w : (1 << 22);   // the kernels' default wait limit
  *skip_tile = g_skip_tile.load(std::memory_order_relaxed);
}

cudaError_t simt_launch_bf16_bf16(const DecodeArgs&, int, cudaStream_t);
cudaError_t simt_launch_f16_f16(const DecodeArgs&, int, cudaStream_t);
cudaError_t simt_launch_q8_0_bf16(const DecodeArgs&, int, cudaStream_t);
cudaError_t simt_launch_q8_0_q8_0(const DecodeArgs&, int, cudaStream_t);
cudaError_t simt_launch_q4s_q4s(const DecodeArgs&, int, cudaStream_t);
cudaError_t simt_launch_q8_0_q4s(const DecodeArgs&, int, cudaStream_t);
cudaError_t simt_launch_q4s_q8_0(const DecodeArgs&, int, cudaStream_t);
cudaError_t simt_launch_q4s_bf16(const DecodeArgs&, int, cudaStream_t);
using MmaFn = cudaError_t (*)(const DecodeArgs&, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
cudaError_t mma_launch_bf16_bf16(const DecodeArgs&, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
cudaError_t mma_launch_f16_f16(const DecodeArgs&, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
cudaError_t mma_launch_q8_0_bf16(const DecodeArgs&, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
cudaError_t mma_launch_q8_0_q8_0(const DecodeArgs&, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
cudaError_t mma_launch_q4s_q4s(const DecodeArgs&, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
cudaError_t mma_launch_q8_0_q4s(const DecodeArgs&, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
cudaError_t mma_launch_q4s_q8_0(const DecodeArgs&, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
cudaError_t mma_launch_q4s_bf16(const DecodeArgs&, int, const CUtensorMap&, const CUtensorMap&, cudaStream_t);
cudaError_t prefill_launch(int kc, int vc, const PrefillArgs& a, int batch, int head_dim,
                           const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream);
int mma_occupancy_bf16_bf16(int, int, int*, int);
int mma_occupancy_f16_f16(int, int, int*, int);
int mma_occupancy_q8_0_bf16(int, int, int*, int);
int mma_occupancy_q8_0_q8_0(int, int, int*, int);
int mma_occupancy_q4s_q4s(int, int, int*, int);
int mma_occupancy_q8_0_q4s(int, int, int*, int);
int mma_occupancy_q4s_q8_0(int, int, int*, int);
int mma_occupancy_q4s_bf16(int, int, int*, int);

namespace {

using SimtFn = cudaError_t (*)(const DecodeArgs&, int, cudaStream_t);

SimtFn simt_fn(int kc, int vc) {
  if (kc == KVQ_CODEC_BF16 && vc == KVQ_CODEC_BF16) return simt_launch_bf16_bf16;
  if (kc == KVQ_CODEC_F16 && vc == KVQ_CODEC_F16) return simt_launch_f16_f16;
  if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_BF16) return simt_launch_q8_0_bf16;
  if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_Q8_0) return simt_launch_q8_0_q8_0;
  if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_Q4S) return simt_launch_q4s_q4s;
  if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_Q4S) return simt_launch_q8_0_q4s;
  if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_Q8_0) return simt_launch_q4s_q8_0;
  if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_BF16) return simt_launch_q4s_bf16;
  return nullptr;
}

MmaFn mma_fn(int kc, int vc) {
  if (kc == KVQ_CODEC_BF16 && vc == KVQ_CODEC_BF16) return mma_launch_bf16_bf16;
  if (kc == KVQ_CODEC_F16 && vc == KVQ_CODEC_F16) return mma_launch_f16_f16;
  if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_BF16) return mma_launch_q8_0_bf16;
  if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_Q8_0) return mma_launch_q8_0_q8_0;
  if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_Q4S) return mma_launch_q4s_q4s;
  if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_Q4S) return mma_launch_q8_0_q4s;
  if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_Q8_0) return mma_launch_q4s_q8_0;
  if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_BF16) return mma_launch_q4s_bf16;
  return nullptr;
}

// Resident CTAs per SM of the tensor-core kernel for this shape, and its pipelines per
// CTA (cached per process).
int mma_occupancy(int kc, int vc, int head_dim, int group, int* pipes, bool solo = false) {
  static std::mutex mu;
  static int cache[4][4][3][5] = {};
  static int cache_pipes[4][4][3][5] = {};
  const int di = head_dim == 64 ? 0 : head_dim == 128 ? 1 : 2;
  const int gi = group <= 4 ? (solo ? 4 : 0) : group <= 8 ? 1 : group <= 16 ? 2 : 3;
  std::lock_guard<std::mutex> lock(mu);
  int& slot = cache[kc & 3][vc & 3][di][gi];
  int& pslot = cache_pipes[kc & 3][vc & 3][di][gi];
  if (slot == 0) {
    int n = 0, np = 1;
    if (kc == KVQ_CODEC_BF16 && vc == KVQ_CODEC_BF16) n = mma_occupancy_bf16_bf16(head_dim, group, &np, solo ? 1 : 0);
    else if (kc == KVQ_CODEC_F16 && vc == KVQ_CODEC_F16) n = mma_occupancy_f16_f16(head_dim, group, &np, solo ? 1 : 0);
    else if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_BF16) n = mma_occupancy_q8_0_bf16(head_dim, group, &np, solo ? 1 : 0);
    else if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_Q8_0) n = mma_occupancy_q8_0_q8_0(head_dim, group, &np, solo ? 1 : 0);
    else if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_Q4S) n = mma_occupancy_q4s_q4s(head_dim, group, &np, solo ? 1 : 0);
    else if (kc == KVQ_CODEC_Q8_0 && vc == KVQ_CODEC_Q4S) n = mma_occupancy_q8_0_q4s(head_dim, group, &np, solo ? 1 : 0);
    else if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_Q8_0) n = mma_occupancy_q4s_q8_0(head_dim, group, &np, solo ? 1 : 0);
    else if (kc == KVQ_CODEC_Q4S && vc == KVQ_CODEC_BF16) n = mma_occupancy_q4s_bf16(head_dim, group, &np, solo ? 1 : 0);
    slot = n > 0 ? n : 1;
    pslot = np > 0 ? np : 1;
  }
  *pipes = pslot;
  return slot;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// TMA map over a store's row data: a 4-D byte tensor {row_bytes, page_size, kv_heads,
// pages} with the slab strides; boxes of 64 rows x min(row_bytes, 128) bytes, swizzled
// over the box width so that ldmatrix reads of 8 consecutive rows hit distinct banks.
bool encode_rows_map(kvq_store* s) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const int rb = s->row_bytes;
  const int line = rb >= 128 ? 128 : rb;
  cuuint64_t dims[4] = {(cuuint64_t)rb, (cuuint64_t)s->desc.page_size, (cuuint64_t)s->desc.num_kv_heads,
                        (cuuint64_t)s->desc.num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)rb, (cuuint64_t)s->slab_bytes,
                           (cuuint64_t)s->slab_bytes * (cuuint64_t)s->desc.num_kv_heads};
  cuuint32_t box[4] = {(cuuint32_t)line, 64u, 1u, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapSwizzle sw = line == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : line == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
  const CUresult r = enc(&s->rows_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, s->buf, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kvq_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return KVQ_OK;
  if (e == cudaErrorNotSupported) return KVQ_ERR_UNSUPPORTED;
  return KVQ_ERR_CUDA;
}

bool desc_ok(const kvq_store_desc* d) {
  if (!d) return false;
  if (d->codec < KVQ_CODEC_BF16 || d->codec > KVQ_CODEC_Q4S) return false;
  if (d->num_kv_heads < 1 || d->num_pages < 1) return false;
  if (d->head_dim != 64 && d->head_dim != 128 && d->head_dim != 256) return false;
  if (d->page_size < 64 || d->page_size > 1024 || d->page_size % 64 != 0) return false;
  return true;
}

size_t desc_bytes(const kvq_store_desc* d) {
  const size_t slab = (size_t)d->page_size *
                      (codec_row_bytes(d->codec, d->head_dim) + 2 * codec_scales(d->codec, d->head_dim));
  return slab * (size_t)d->num_kv_heads * (size_t)d->num_pages;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Plan {
  int chunk_tokens;
  int n_chunks;
  int n_groups;
  int variant;
  int records;       // record mode: records per (sequence, KV head), else 0
  bool solo;         // tensor-core kernel, at most 4 rows per KV head: one pipeline per CTA
  size_t ml_off;     // chunk partials: o at 0, (m, l) at ml_off
  size_t go_off;     // group partials: o at go_off, (m, l) at gml_off
  size_t gml_off;
  size_t cnt_off;    // unit counters, then group counters, then sequence counters
  size_t seq_cnt_off;
  size_t total;
};

// Split planner (step a2).  A pure function of its arguments and the device (SM count,
// resident CTAs per SM of the chosen kernel).  The default split gives each (sequence,
// KV head) n_chunks = slots / units CTAs, where slots = SMs x resident CTAs per SM and
// units = batch x kv_heads, so the longest sequence fills one wave; chunk_tokens =
// ceil(max_len / n_chunks) rounded up to 64 is the number of tokens a CTA covers (the
// tensor-core kernel deals the 64-token tiles to its CTAs round-robin).  When units
// outnumber slots, chunks are capped (1024 tokens per pipeline, 2048 for single-pipeline CTAs)
// so long sequences still spread.
// It sizes the workspace: chunk partials, group partials (groups of kMergeGroup chunks)
// and the arrival counters of the merge.
kvq_status make_plan(const kvq_store* k, const kvq_store* v, int batch, int num_q_heads,
                     int max_len_hint, const kvq_decode_opts* opts, Plan* p) {
  const int hint = max_len_hint > 0 ? max_len_hint : 1;
  int chunk = opts ? opts->chunk_tokens : 0;
  if (chunk < 0 || chunk % 64 != 0) return KVQ_ERR_INVALID_ARG;
  p->variant = (opts && opts->variant) ? opts->variant : 2;
  const int group_all = num_q_heads / k->desc.num_kv_heads;
  const int sms = sm_count();
  if (sms <= 0) return KVQ_ERR_CUDA;
  // More (sequence, KV head) units than SMs: many CTAs, each short (batched decode); the
  // single-pipeline configuration keeps four of them per SM so that their prologues and
  // merges overlap.  Also from 9 units up where whole single-pipeline CTAs per unit fill at
  // least 90 % of the 4 x SMs slots in one wave: a unit's CTAs then come in steps of one
  // pipeline instead of four (4 sequences x 65536 tokens 130 -> 117 us, 8 x 32768 141 ->
  // 123 us).  Otherwise one CTA of four pipelines per SM.
  const long long units_all = (long long)batch * k->desc.num_kv_heads;
  const int vcodec = v ? v->desc.codec : k->desc.codec;
  bool solo_ok = p->variant == 2 && group_all <= 4 && k->desc.head_dim <= 128;
  long long solo_slots = 0;
  if (solo_ok) {
    int solo_pipes = 1;
    solo_slots = (long long)sms * mma_occupancy(k->desc.codec, vcodec, k->desc.head_dim, group_all, &solo_pipes, true);
    solo_ok = solo_slots > 0;
  }
  const bool solo_fills = solo_ok && units_all > 8 && (solo_slots / units_all) * units_all * 10 >= 9 * solo_slots;
  p->solo = solo_ok && (units_all > sms || solo_fills);
  int pipes = 1;
  if (p->variant == 2)
    (void)mma_occupancy(k->desc.codec, v ? v->desc.codec : k->desc.codec, k->desc.head_dim, group_all, &pipes,
                        p->solo);
  if (chunk == 0) {
    const int group = num_q_heads / k->desc.num_kv_heads;
    const int per_sm = p->variant == 2 ? mma_occupancy(k->desc.codec, v ? v->desc.codec : k->desc.codec,
                                                       k->desc.head_dim, group, &pipes, p->solo)
                                       : 2;
    const long long units = (long long)batch * k->desc.num_kv_heads;
    const long long slots = (long long)sms * per_sm;
    long long want = slots >= units ? slots / units : 1;   // chunks per unit
    const long long max_chunks = (hint + 127) / 128;           // >= 128 tokens per chunk
    if (want > max_chunks) want = max_chunks;
    long long c = (hint + want - 1) / want;
    c = (c + 63) / 64 * 64;
    if (c < 128) c = 128;
    // With one or two CTAs per unit a long sequence among short ones would run alone
    // (lengths are on the device): keep chunks short enough for the block scheduler to
    // balance the batch (1024 tokens per pipeline of the CTA; 2048 for the single-pipeline
    // CTAs of a batch, whose fixed costs 1024-token chunks did not amortize: the
    // 64-sequence ragged batch 496 -> 449 us, uniform batches unchanged or faster).
    const long long cap_tokens = (p->solo ? 2048LL : 1024LL) * pipes;
    const bool capped = units * 4 > slots && c > cap_tokens;
    if (capped) c = cap_tokens;
    chunk = (int)c;
    // One full wave: `want` chunks per unit even where rounding the chunk up to whole
    // tiles would need fewer (the tensor-core kernel deals tiles round-robin, so every
    // resident slot gets work; chunk_tokens then only bounds the length)
    p->n_chunks = capped ? (int)((hint + c - 1) / c) : (int)want;
  } else {
    p->n_chunks = (hint + chunk - 1) / chunk;
  }
  p->chunk_tokens = chunk;
  p->n_groups = (p->n_chunks + kMergeGroup - 1) / kMergeGroup;
  const size_t D = (size_t)k->desc.head_dim;
  const size_t heads = (size_t)batch * num_q_heads;
  const size_t units = (size_t)batch * k->desc.num_kv_heads;
  // Record mode (tensor-core kernel, at most 4 query rows per KV head, head_dim <= 128,
  // four-pipeline CTAs): every warp leaves its partial as a record ((chunk * pipes + pipe)
  // * 4 + slice) and a separate merge kernel combines them.  Used while all records fit in
  // 16 MiB (they stay in L2 between the two kernels and add little traffic); otherwise,
  // beyond 4096 records per unit, and for the single-pipeline CTAs of a batch (many units
  // of few chunks, where a second kernel over every unit cost more than it saved: 160 ->
  // 150 us for 160 sequences of 2048 tokens), the decode kernel merges in place
  // (last-arriving CTA; a unit of one chunk writes its output directly).
  const long long recs = (long long)p->n_chunks * pipes * 4;
  const long long rec_bytes = (long long)units * recs * (long long)(D * 4 + 8) * 4;
  p->records = (p->variant == 2 && !p->solo && group_all <= 4 && D <= 128 && recs <= 4096 &&
                rec_bytes <= (16LL << 20)) ? (int)recs : 0;
  if (p->records) {
    p->ml_off = round_up(units * p->records * (D * 4) * sizeof(float), 256);
    p->go_off = p->ml_off + round_up(units * p->records * 8 * sizeof(float), 256);
    p->gml_off = p->go_off;
    p->cnt_off = p->gml_off;
    p->seq_cnt_off = p->cnt_off + units * (1 + p->n_groups) * sizeof(unsigned);
    p->total = p->cnt_off + round_up((units * (1 + p->n_groups) + (size_t)batch) * sizeof(unsigned), 256);
    return KVQ_OK;
  }
  p->ml_off = round_up(heads * p->n_chunks * D * sizeof(float), 256);
  p->go_off = p->ml_off + round_up(heads * p->n_chunks * 2 * sizeof(float), 256);
  p->gml_off = p->go_off + round_up(heads * p->n_groups * D * sizeof(float), 256);
  p->cnt_off = p->gml_off + round_up(heads * p->n_groups * 2 * sizeof(float), 256);
  p->seq_cnt_off = p->cnt_off + units * (1 + p->n_groups) * sizeof(unsigned);
  p->total = p->cnt_off + round_up((units * (1 + p->n_groups) + (size_t)batch) * sizeof(unsigned), 256);
  return KVQ_OK;
}

}  // namespace

// Workspace size of a decode call and the offset of its arrival counters (the part a
// reused workspace must have zeroed before a call).
kvq_status decode_workspace_layout(const kvq_store* k_store, const kvq_store* v_store, int batch,
                                   int num_q_heads, int max_len_hint, const kvq_decode_opts* opts,
                                   size_t* total, size_t* counters_off) {
  if (!k_store || !v_store || batch < 1 || num_q_heads < 1 || max_len_hint < 0) return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % k_store->desc.num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  Plan p;
  const kvq_status st = make_plan(k_store, v_store, batch, num_q_heads, max_len_hint, opts, &p);
  if (st != KVQ_OK) return st;
  *total = p.total;
  *counters_off = p.cnt_off;
  return KVQ_OK;
}

}  // namespace kvq

using namespace kvq;

extern "C" {

kvq_status kvq_store_bytes(const kvq_store_desc* desc, size_t* bytes) {
  if (!desc_ok(desc) || !bytes) return KVQ_ERR_INVALID_ARG;
  *bytes = desc_bytes(desc);
  return KVQ_OK;
}

kvq_status kvq_store_create(const kvq_store_desc* desc, void* buf, size_t buf_bytes,
                            kvq_store** out) {
  if (!out) return KVQ_ERR_INVALID_ARG;
  *out = nullptr;
  if (!desc_ok(desc) || !buf || !aligned(buf, 256)) return KVQ_ERR_INVALID_ARG;
  if (buf_bytes < desc_bytes(desc)) return KVQ_ERR_INVALID_ARG;
  kvq_store* s = new (std::nothrow) kvq_store();
  if (!s) return KVQ_ERR_INVALID_ARG;
  s->desc = *desc;
  s->buf = static_cast<uint8_t*>(buf);
  s->bytes = buf_bytes;
  s->row_bytes = codec_row_bytes(desc->codec, desc->head_dim);
  s->n_scales = codec_scales(desc->codec, desc->head_dim);
  s->slab_bytes = (long long)desc->page_size * (s->row_bytes + 2 * s->n_scales);
  s->rows_map_ok = encode_rows_map(s);
  if (cudaGetDevice(&s->device) != cudaSuccess ||
      cudaMalloc(reinterpret_cast<void**>(&s->status), sizeof(int32_t)) != cudaSuccess) {
    delete s;
    return KVQ_ERR_CUDA;
  }
  if (cudaMemset(s->status, 0, sizeof(int32_t)) != cudaSuccess) {
    cudaFree(s->status);
    delete s;
    return KVQ_ERR_CUDA;
  }
  *out = s;
  return KVQ_OK;
}

kvq_status kvq_destroy(kvq_store* store) {
  if (!store) return KVQ_OK;
  const cudaError_t e = cudaFree(store->status);
  delete store;
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_append(kvq_store* store, const void* rows, int n_new, int batch,
                      const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                      void* stream) {
  if (!store || !seq_lens || !page_table || batch < 1 || n_new < 0 || max_pages < 1)
    return KVQ_ERR_INVALID_ARG;
  if (n_new == 0) return KVQ_OK;
  if (!rows || !aligned(rows, 16)) return KVQ_ERR_INVALID_ARG;
  return from_cuda(launch_append(store, static_cast<const __nv_bfloat16*>(rows), n_new, batch,
                                 seq_lens, page_table, max_pages, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_append_kv(kvq_store* k_store, kvq_store* v_store, const void* k_rows, const void* v_rows,
                         int n_new, int batch, int32_t* seq_lens, const int32_t* page_table, int max_pages,
                         int advance, void* stream) {
  if (!k_store || !v_store || !seq_lens || !page_table || batch < 1 || n_new < 0 || max_pages < 1)
    return KVQ_ERR_INVALID_ARG;
  const kvq_store_desc& kd = k_store->desc;
  const kvq_store_desc& vd = v_store->desc;
  if (kd.num_kv_heads != vd.num_kv_heads || kd.head_dim != vd.head_dim || kd.page_size != vd.page_size)
    return KVQ_ERR_INVALID_ARG;
  if (n_new == 0) return KVQ_OK;
  if (!k_rows || !v_rows || !aligned(k_rows, 16) || !aligned(v_rows, 16)) return KVQ_ERR_INVALID_ARG;
  return from_cuda(launch_append_kv(k_store, v_store, static_cast<const __nv_bfloat16*>(k_rows),
                                    static_cast<const __nv_bfloat16*>(v_rows), n_new, batch, seq_lens, page_table,
                                    max_pages, advance ? 1 : 0, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_seq_lens_add(int32_t* seq_lens, int batch, int n, void* stream) {
  if (!seq_lens || batch < 1) return KVQ_ERR_INVALID_ARG;
  return from_cuda(launch_seq_lens_add(seq_lens, batch, n, static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_decode_workspace_bytes(const kvq_store* k_store, const kvq_store* v_store,
                                      int batch, int num_q_heads, int max_len_hint,
                                      const kvq_decode_opts* opts, size_t* bytes) {
  if (!k_store || !v_store || !bytes || batch < 1 || num_q_heads < 1 || max_len_hint < 0)
    return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % k_store->desc.num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  Plan p;
  const kvq_status st = make_plan(k_store, v_store, batch, num_q_heads, max_len_hint, opts, &p);
  if (st != KVQ_OK) return st;
  *bytes = p.total;
  return KVQ_OK;
}

kvq_status kvq_pointer_kind(const void* p, int32_t* kind) {
  if (!p || !kind) return KVQ_ERR_INVALID_ARG;
  cudaPointerAttributes at = {};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    (void)cudaGetLastError();   // clear the sticky-free error of the query
    *kind = -1;
    return KVQ_OK;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) *kind = 0;
  else if (at.type == cudaMemoryTypeHost && at.devicePointer == p) *kind = 1;
  else *kind = -1;
  return KVQ_OK;
}

kvq_status kvq_decode_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (!workspace || workspace_bytes == 0) return KVQ_ERR_INVALID_ARG;
  return from_cuda(cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace kvq {
namespace {

// kvq_flash_decode, and with k_new set the fused append step (kvq_flash_decode_append).
// With reset_counters the workspace's counters are zeroed on the stream right before the
// launch, after every check has passed (the fixed-array entry point's workspace keeps the
// previous call's contents).
kvq_status decode_impl(const void* q, const void* k_new, const void* v_new, const kvq_store* k_store,
                       const kvq_store* v_store, const int32_t* seq_lens, int32_t* seq_lens_adv,
                       const int32_t* page_table, int max_pages, kvq_codec codec, float* out,
                       int batch, int num_q_heads, int tokens, float softmax_scale, int max_len_hint,
                       const kvq_decode_opts* opts, void* workspace, size_t workspace_bytes,
                       void* stream, bool reset_counters = false) {
  if (!q || !k_store || !v_store || !seq_lens || !page_table || !out || !workspace)
    return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || num_q_heads < 1 || tokens < 1 || max_pages < 1 || max_len_hint < 0)
    return KVQ_ERR_INVALID_ARG;
  const kvq_store_desc& kd = k_store->desc;
  const kvq_store_desc& vd = v_store->desc;
  if (kd.num_kv_heads != vd.num_kv_heads || kd.head_dim != vd.head_dim ||
      kd.page_size != vd.page_size || kd.num_pages != vd.num_pages)
    return KVQ_ERR_INVALID_ARG;
  if (codec.k != kd.codec || codec.v != vd.codec) return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % kd.num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if ((long long)max_len_hint > (long long)max_pages * kd.page_size) return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16) || !aligned(workspace, 16)) return KVQ_ERR_INVALID_ARG;
  if (k_new && (!v_new || !aligned(k_new, 16) || !aligned(v_new, 16))) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if ((long long)num_q_heads * tokens > (1 << 24)) return KVQ_ERR_INVALID_ARG;
  // the kernels see tokens x heads query rows: row (h, i) of a KV head's group is virtual
  // head h * tokens + i, which is where [B][Hq][tokens][D] puts it
  const int rows = num_q_heads * tokens;
  const int group = rows / kd.num_kv_heads;
  Plan p;
  kvq_status st = make_plan(k_store, v_store, batch, rows, max_len_hint, opts, &p);
  if (st != KVQ_OK) return st;
  if (workspace_bytes < p.total) return KVQ_ERR_WORKSPACE;
  // query rows per KV head: up to 16, or 32 for q8_0 K and V at head_dim >= 128 (the
  // tensor-core kernel's heads-on-M loop)
  const bool rows32 = kd.codec == KVQ_CODEC_Q8_0 && vd.codec == KVQ_CODEC_Q8_0 && kd.head_dim >= 128;
  if (group > (rows32 && p.variant == 2 ? 32 : 16) || p.variant < 1 || p.variant > 2) return KVQ_ERR_UNSUPPORTED;
  if ((k_new || tokens > 1) && p.variant != 2) return KVQ_ERR_UNSUPPORTED;
  SimtFn sfn = simt_fn(kd.codec, vd.codec);
  MmaFn mfn = mma_fn(kd.codec, vd.codec);
  if (p.variant == 1 && !sfn) return KVQ_ERR_UNSUPPORTED;
  if (p.variant == 2 && (!mfn || !k_store->rows_map_ok || !v_store->rows_map_ok)) return KVQ_ERR_UNSUPPORTED;

  DecodeArgs a = {};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = view_of(k_store);
  a.v = view_of(v_store);
  a.seq_lens = seq_lens;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.batch = batch;
  a.num_q_heads = rows;
  a.group = group;
  a.tokens = tokens;
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt((float)kd.head_dim);
  a.qk_scale_log2 = scale * 1.4426950408889634f;
  a.chunk_tokens = p.chunk_tokens;
  a.n_chunks = p.n_chunks;
  a.part_o = static_cast<float*>(workspace);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  a.part_ml = reinterpret_cast<float*>(ws + p.ml_off);
  a.gpart_o = reinterpret_cast<float*>(ws + p.go_off);
  a.gpart_ml = reinterpret_cast<float*>(ws + p.gml_off);
  a.n_groups = p.n_groups;
  a.counters = reinterpret_cast<unsigned*>(ws + p.cnt_off);
  a.grp_counter_off = (long long)batch * kd.num_kv_heads;
  a.out = out;
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.seq_lens_adv = seq_lens_adv;
  a.seq_counters = reinterpret_cast<unsigned*>(ws + p.seq_cnt_off);
  a.warp_records = p.records;
  a.solo = p.solo ? 1 : 0;
  // the heads-on-M loop (q8_0 K and V, head_dim 128 or 256, 9..32 query rows per KV head)
  // leaves its chunk partials to the chunk merge kernel
  a.chunk_merge = (p.variant == 2 && kd.codec == KVQ_CODEC_Q8_0 && vd.codec == KVQ_CODEC_Q8_0 &&
                   (kd.head_dim == 128 || kd.head_dim == 256) && group > 8 && p.n_chunks > 1)
                      ? 1 : 0;
  fault_injection(&a.wait_limit, &a.skip_tile);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (reset_counters && cudaMemsetAsync(ws + p.cnt_off, 0, p.total - p.cnt_off, s) != cudaSuccess)
    return KVQ_ERR_CUDA;
  if (p.variant == 2) {
    // the tensor-core kernel merges the split itself (last CTA per unit), or leaves its
    // partials to a merge kernel launched right after it (record and chunk-merge modes)
    st = from_cuda(mfn(a, kd.head_dim, k_store->rows_map, v_store->rows_map, s));
    if (st != KVQ_OK) return st;
    if (a.chunk_merge) return from_cuda(launch_chunk_merge_pdl(a, kd.head_dim, s));
    if (!p.records) return st;
    return from_cuda(launch_record_merge_pdl(a, kd.head_dim, vd.codec, s));
  }
  st = from_cuda(sfn(a, kd.head_dim, s));
  if (st != KVQ_OK) return st;
  return from_cuda(launch_combine_pdl(a, kd.head_dim, s));
}

}  // namespace

kvq_status decode_reset(const void* q, const kvq_store* k_store, const kvq_store* v_store,
                        const int32_t* seq_lens, const int32_t* page_table, int max_pages, kvq_codec codec,
                        float* out, int batch, int num_q_heads, float softmax_scale, int max_len_hint,
                        const kvq_decode_opts* opts, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(q, nullptr, nullptr, k_store, v_store, seq_lens, nullptr, page_table, max_pages, codec,
                     out, batch, num_q_heads, 1, softmax_scale, max_len_hint, opts, workspace, workspace_bytes,
                     stream, true);
}

}  // namespace kvq

extern "C" {

kvq_status kvq_flash_decode(const void* q, const kvq_store* k_store, const kvq_store* v_store,
                            const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                            kvq_codec codec, float* out, int batch, int num_q_heads,
                            float softmax_scale, int max_len_hint,
                            const kvq_decode_opts* opts, void* workspace,
                            size_t workspace_bytes, void* stream) {
  return decode_impl(q, nullptr, nullptr, k_store, v_store, seq_lens, nullptr, page_table, max_pages,
                     codec, out, batch, num_q_heads, 1, softmax_scale, max_len_hint, opts, workspace,
                     workspace_bytes, stream);
}

kvq_status kvq_flash_decode_multi(const void* q, const kvq_store* k_store, const kvq_store* v_store,
                                  const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                                  kvq_codec codec, float* out, int batch, int num_q_heads, int num_tokens,
                                  float softmax_scale, int max_len_hint, const kvq_decode_opts* opts,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(q, nullptr, nullptr, k_store, v_store, seq_lens, nullptr, page_table, max_pages,
                     codec, out, batch, num_q_heads, num_tokens, softmax_scale, max_len_hint, opts,
                     workspace, workspace_bytes, stream);
}

kvq_status kvq_flash_decode_append(const void* q, const void* k_new, const void* v_new,
                                   kvq_store* k_store, kvq_store* v_store, int32_t* seq_lens,
                                   const int32_t* page_table, int max_pages, kvq_codec codec,
                                   float* out, int batch, int num_q_heads, float softmax_scale,
                                   int max_len_hint, int advance, const kvq_decode_opts* opts,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  if (!k_new || !v_new) return KVQ_ERR_INVALID_ARG;
  return decode_impl(q, k_new, v_new, k_store, v_store, seq_lens, advance ? seq_lens : nullptr,
                     page_table, max_pages, codec, out, batch, num_q_heads, 1, softmax_scale,
                     max_len_hint, opts, workspace, workspace_bytes, stream);
}

kvq_status kvq_prefill_attention(const void* q, const kvq_store* k_store, const kvq_store* v_store,
                                 const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                                 kvq_codec codec, float* out, int batch, int num_q_heads,
                                 int num_tokens, float softmax_scale, void* stream) {
  if (!q || !k_store || !v_store || !seq_lens || !page_table || !out) return KVQ_ERR_INVALID_ARG;
  if (batch < 1 || num_q_heads < 1 || num_tokens < 1 || max_pages < 1) return KVQ_ERR_INVALID_ARG;
  const kvq_store_desc& kd = k_store->desc;
  const kvq_store_desc& vd = v_store->desc;
  if (kd.num_kv_heads != vd.num_kv_heads || kd.head_dim != vd.head_dim ||
      kd.page_size != vd.page_size || kd.num_pages != vd.num_pages)
    return KVQ_ERR_INVALID_ARG;
  if (codec.k != kd.codec || codec.v != vd.codec) return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % kd.num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(out, 16)) return KVQ_ERR_INVALID_ARG;
  if (!std::isfinite(softmax_scale)) return KVQ_ERR_INVALID_ARG;
  if ((long long)num_tokens * num_q_heads > (1LL << 30)) return KVQ_ERR_INVALID_ARG;
  if (!k_store->rows_map_ok || !v_store->rows_map_ok) return KVQ_ERR_UNSUPPORTED;
  PrefillArgs a = {};
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.k = view_of(k_store);
  a.v = view_of(v_store);
  a.seq_lens = seq_lens;
  a.page_table = page_table;
  a.max_pages = max_pages;
  a.num_q_heads = num_q_heads;
  a.group = num_q_heads / kd.num_kv_heads;
  a.tokens = num_tokens;
  const float scale = softmax_scale > 0.0f ? softmax_scale : 1.0f / std::sqrt((float)kd.head_dim);
  a.qk_scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  fault_injection(&a.wait_limit, &a.skip_tile);
  const cudaError_t e = prefill_launch(kd.codec, vd.codec, a, batch, kd.head_dim, k_store->rows_map,
                                       v_store->rows_map, static_cast<cudaStream_t>(stream));
  return e == cudaErrorNotSupported ? KVQ_ERR_UNSUPPORTED : from_cuda(e);
}

kvq_status kvq_dequantize(const kvq_store* src, kvq_store* dst, const int32_t* seq_lens,
                          const int32_t* page_table, int max_pages, int batch, void* stream) {
  if (!src || !dst || !seq_lens || !page_table || batch < 1 || max_pages < 1) return KVQ_ERR_INVALID_ARG;
  const kvq_store_desc& sd = src->desc;
  const kvq_store_desc& dd = dst->desc;
  if (sd.num_kv_heads != dd.num_kv_heads || sd.head_dim != dd.head_dim || sd.page_size != dd.page_size ||
      sd.num_pages != dd.num_pages)
    return KVQ_ERR_INVALID_ARG;
  if ((sd.codec != KVQ_CODEC_Q8_0 && sd.codec != KVQ_CODEC_Q4S) ||
      (dd.codec != KVQ_CODEC_F16 && dd.codec != KVQ_CODEC_BF16))
    return KVQ_ERR_UNSUPPORTED;
  return from_cuda(launch_dequantize(src, dst, seq_lens, page_table, max_pages, batch,
                                     static_cast<cudaStream_t>(stream)));
}

kvq_status kvq_store_get_error(kvq_store* store, int32_t* device_code) {
  if (!store || !device_code) return KVQ_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaMemcpy(&v, store->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return KVQ_ERR_CUDA;
  if (cudaMemset(store->status, 0, sizeof(int32_t)) != cudaSuccess) return KVQ_ERR_CUDA;
  *device_code = v;
  return v ? KVQ_ERR_DEVICE_FAULT : KVQ_OK;
}

uint64_t kvq_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

kvq_status kvq_set_fault_injection(int32_t wait_limit, int32_t skip_tile) {
  if (wait_limit < 0 || skip_tile < -1) return KVQ_ERR_INVALID_ARG;
  kvq::g_wait_limit.store(wait_limit, std::memory_order_relaxed);
  kvq::g_skip_tile.store(skip_tile, std::memory_order_relaxed);
  return KVQ_OK;
}

const char* kvq_status_string(kvq_status status) {
  switch (status) {
    case KVQ_OK: return "KVQ_OK";
    case KVQ_ERR_INVALID_ARG: return "KVQ_ERR_INVALID_ARG";
    case KVQ_ERR_UNSUPPORTED: return "KVQ_ERR_UNSUPPORTED";
    case KVQ_ERR_CUDA: return "KVQ_ERR_CUDA";
    case KVQ_ERR_DEVICE_FAULT: return "KVQ_ERR_DEVICE_FAULT";
    case KVQ_ERR_WORKSPACE: return "KVQ_ERR_WORKSPACE";
    default: return "KVQ_UNKNOWN_STATUS";
  }
}

}  // extern "C"
