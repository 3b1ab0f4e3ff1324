/*
 * kvq.h -- C ABI of a fused dequant-on-load flash-decode library for a resident,
 * paged, block-quantized KV cache (NVIDIA GB300, sm_103a).
 *
 * What it computes.  Single-token decode attention (split-K flash-decode) that reads
 * the quantized KV store directly and dequantizes inside the kernel, the
 * "flash-decode-over-quant" class that rMLX issue #292 ("Root cause", correction)
 * names as the target, with the "dequantize KV on load" treatment of halobench record
 * clm-0022 (METHOD) and a 16-bit KV arm kept as the control (that record credits its
 * speedup to the quantized arm because the f16 arm did not move).  The prefix stays
 * resident on the device and new rows are encoded there,
 * so no step restages the prefix through the host (rMLX issue #295, "Root cause" and
 * "Fix direction").
 *
 * Conventions for every call below.
 *  - All pointers named "device" are CUDA device pointers on the current device; all
 *    others are host pointers.  The library never frees memory it did not allocate.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Every call that takes a stream only enqueues work on it and returns; none waits
 *    for the device, except kvq_store_get_error.
 *  - Shapes, codecs, alignment and null pointers are checked on the host before any
 *    work is enqueued; a failed check returns KVQ_ERR_INVALID_ARG or
 *    KVQ_ERR_UNSUPPORTED and enqueues nothing.
 *  - Bad values found in device data (a page id outside [0, num_pages), a position past
 *    the page table, a negative or too-long sequence length) never trap: the kernel
 *    skips the affected row or tile and records the first such fault in the store's
 *    device status word, read back by kvq_store_get_error.
 *  - A CUDA launch failure returns KVQ_ERR_CUDA.
 *
 * Store layout (one store holds either K or V of every layer-head it was sized for):
 *   num_pages pages x num_kv_heads slabs; slab (page, head) =
 *     [page_size rows x row_bytes]            row data, token-major
 *     [page_size rows x (head_dim/32) x fp16]  block scales (q8_0 and q4s only)
 *   row_bytes = 2*head_dim (bf16, f16), head_dim (q8_0), head_dim/2 (q4s).
 *   Token position pos of sequence b lives in physical page
 *   page_table[b*max_pages + pos/page_size], row pos % page_size.
 *
 * Codecs (blocks of 32 consecutive elements along head_dim; inputs are bf16):
 *   amax = max|x|; d = fp16_rn(amax / c) (fp32 quotient); q = 0 if d == 0, else
 *   clamp(round_half_away(x / d) (fp32 quotient), -c, c); c = 127 (q8_0) or 7 (q4s).
 *   q8_0 stores int8 q; q4s stores u = q + 8 as nibbles, element 2k in the low nibble
 *   of block byte k.  bf16 stores the input bits; f16 stores fp16_rn(x).
 *   Dequantized value: d * q.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1,   /* bad pointer, shape, size or alignment */
  KVQ_ERR_UNSUPPORTED = 2,   /* valid but not built: codec pair, head_dim, group size */
  KVQ_ERR_CUDA = 3,          /* a CUDA runtime call or kernel launch failed */
  KVQ_ERR_DEVICE_FAULT = 4,  /* kvq_store_get_error: a kernel recorded a data fault */
  KVQ_ERR_WORKSPACE = 5      /* the workspace passed is smaller than required */
} kvq_status;

typedef enum kvq_codec_id {
  KVQ_CODEC_BF16 = 0,        /* 16-bit control arm, bf16 values as given */
  KVQ_CODEC_F16 = 1,         /* 16-bit control arm, fp16_rn of the bf16 input */
  KVQ_CODEC_Q8_0 = 2,        /* 8-bit symmetric blocks of 32, fp16 scale */
  KVQ_CODEC_Q4S = 3          /* 4-bit symmetric blocks of 32, fp16 scale, q in [-7, 7] */
} kvq_codec_id;

/* Device fault codes recorded in a store's status word (first fault wins). */
enum {
  KVQ_DEVICE_OK = 0,
  KVQ_DEVICE_BAD_PAGE = 1,      /* page id outside [0, num_pages) */
  KVQ_DEVICE_BAD_POSITION = 2,  /* append position outside [0, max_pages*page_size) */
  KVQ_DEVICE_BAD_SEQ_LEN = 3,   /* sequence length < 0, past the page table, or past
                                   the max_len_hint that sized the decode split */
  KVQ_DEVICE_TIMEOUT = 4,       /* a kernel's bounded wait for its own tile copies ran
                                   out; the kernel stopped and its outputs are invalid */
  KVQ_DEVICE_BAD_WORKSPACE = 5  /* the workspace's arrival counters were not zero at the
                                   start of a decode (see kvq_decode_workspace_init) */
};

/* Shape of one store.  head_dim in {64, 128, 256}; page_size a multiple of 64 in
 * [64, 1024]; num_kv_heads >= 1; num_pages >= 1. */
typedef struct kvq_store_desc {
  int32_t codec;             /* kvq_codec_id */
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;         /* tokens per page */
  int32_t num_pages;
} kvq_store_desc;

/* Codec pair a decode call expects; must equal the codecs of the stores passed.
 * Built pairs (K/V): bf16/bf16, f16/f16 (16-bit controls), q8_0/bf16 (K-only
 * quantization), q8_0/q8_0, q4s/q4s, q8_0/q4s, q4s/q8_0, q4s/bf16 (the mixed K/V precision
 * families of rMLX issue #292, correction table); others give KVQ_ERR_UNSUPPORTED. */
typedef struct kvq_codec {
  int32_t k;                 /* kvq_codec_id of the K store */
  int32_t v;                 /* kvq_codec_id of the V store */
} kvq_codec;

/* Optional decode settings (pass NULL for the defaults). */
typedef struct kvq_decode_opts {
  int32_t chunk_tokens;      /* split-K chunk length in tokens; 0 = planner's choice.
                                Must be a positive multiple of 64 otherwise. */
  int32_t variant;           /* 0 = auto, 1 = CUDA-core kernel, 2 = tensor-core kernel */
} kvq_decode_opts;

typedef struct kvq_store kvq_store;  /* opaque handle: host metadata + a device status word */

/* Bytes of device memory a store with this shape needs (num_pages * num_kv_heads *
 * page_size * (row_bytes + 2*head_dim/32 for quantized codecs)).  Pure host call.
 * Source: the resident packed store of rMLX issue #295 ("Fix direction": keep the prefix
 * on the device across decode steps and read the quant store directly).  The pages give
 * no API for it; sizing, wrapping caller memory and releasing the handle is the plainest
 * lifecycle that lets the caller (torch) own every byte of device memory. */
kvq_status kvq_store_bytes(const kvq_store_desc* desc, size_t* bytes);

/* Wrap caller-owned device memory `buf` (at least kvq_store_bytes bytes, 256-byte
 * aligned) as a store (the resident store of rMLX issue #295, "Fix direction").  The
 * buffer's previous contents are kept; rows that were never appended hold whatever the
 * buffer held.  Allocates the handle on the host and a 4-byte status word on the current
 * device.  `*out` is valid until kvq_destroy.  Errors: KVQ_ERR_INVALID_ARG for a bad
 * descriptor or a null, unaligned or too small buffer; KVQ_ERR_CUDA when the status word
 * cannot be allocated or cleared (nothing is kept, *out stays NULL). */
kvq_status kvq_store_create(const kvq_store_desc* desc, void* buf, size_t buf_bytes,
                            kvq_store** out);

/* Free the handle and its status word (end of the resident store's life, rMLX issue
 * #295 "Fix direction").  Does not touch `buf`.  The caller must make sure no enqueued
 * work still uses the store.  NULL is accepted.  KVQ_ERR_CUDA if cudaFree fails (the
 * host handle is freed regardless). */
kvq_status kvq_destroy(kvq_store* store);

/* Encode new rows into the store, on the device (a1: on-device encode of new K/V rows;
 * rMLX issue #295 "Fix direction").
 *   rows       device bf16 [batch][n_new][num_kv_heads][head_dim], contiguous, 16-byte aligned.
 *   seq_lens   device int32 [batch]: row i of sequence b is written at position
 *              seq_lens[b] + i.  Not modified (see kvq_seq_lens_add).
 *   page_table device int32 [batch][max_pages].
 * Rows whose position or page is invalid are skipped and recorded as device faults. */
kvq_status kvq_append(kvq_store* store, const void* rows, int n_new, int batch,
                      const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                      void* stream);

/* kvq_append for the K and the V rows of a step in one launch (rows as for kvq_append,
 * k_rows into k_store and v_rows into v_store, both at seq_lens[b] + i).  With
 * advance != 0, seq_lens[b] += n_new afterwards, in stream order, so a decode step is
 * kvq_append_kv + kvq_flash_decode.  The stores must share num_kv_heads, head_dim and
 * page_size; faults are recorded in the store being written. */
kvq_status kvq_append_kv(kvq_store* k_store, kvq_store* v_store, const void* k_rows,
                         const void* v_rows, int n_new, int batch, int32_t* seq_lens,
                         const int32_t* page_table, int max_pages, int advance, void* stream);

/* seq_lens[b] += n for b < batch, on the device (after the K and the V append).  Source:
 * rMLX issue #295 ("Fix direction": no per-step host restage), so the lengths that
 * locate the new rows advance on the device too, in stream order, without a host round
 * trip.  seq_lens: device int32 [batch], caller-owned.  KVQ_ERR_INVALID_ARG for a null
 * pointer or batch < 1; KVQ_ERR_CUDA for a failed launch. */
kvq_status kvq_seq_lens_add(int32_t* seq_lens, int batch, int n, void* stream);

/* Separate dequantize pass (the comparison arm of halobench record clm-0022, METHOD and
 * depth tables: the quantized cache converted outside the attention kernel, then read
 * by a 16-bit decode).  Rewrites rows [0, seq_lens[b]) of every sequence of `src`
 * (q8_0 or q4s) into `dst` (f16 or bf16) at the same positions: value = d * q rounded
 * once to the 16-bit type (d * q is exact in fp32).  The stores must share num_kv_heads,
 * head_dim, page_size and num_pages; page_table and seq_lens as for kvq_append.
 * A length past the table or a bad page id is recorded in dst's status word (rows of
 * that page are skipped).  Not part of the fused path: kvq_flash_decode reads `src`
 * directly. */
kvq_status kvq_dequantize(const kvq_store* src, kvq_store* dst, const int32_t* seq_lens,
                          const int32_t* page_table, int max_pages, int batch, void* stream);

/* Read-only bandwidth probe (a measurement utility, not a step of the method): reads the
 * `bytes` (>= 16, 16-byte aligned start; a tail below 16 bytes is not read) of device
 * buffer `buf` once with streaming 16-byte loads from one full wave of CTAs.  `sink` is a
 * device uint32 the kernel may increment (never for real data).  Time it with events on
 * `stream` to get the achievable read bandwidth that the decode's effective KV GB/s is
 * compared with. */
kvq_status kvq_read_probe(const void* buf, size_t bytes, void* sink, void* stream);

/* Device workspace bytes a kvq_flash_decode (or kvq_flash_decode_append) call with the
 * same stores, batch, head count, max_len_hint and options needs (the split depends on
 * both stores' codecs).  Source: the split-K form of the flash-decode-over-quant kernel
 * class (rMLX issue #292, "Root cause" and its correction): each chunk of the KV length
 * leaves a partial (running max m, sum l, accumulator) that the combine step merges,
 * and those partials live here.  Pure host call; KVQ_ERR_INVALID_ARG for null pointers,
 * batch or head counts < 1, a negative hint or heads not divisible by num_kv_heads.  The workspace holds the split-K partials and, at its end,
 * arrival counters: per (sequence, KV head), per group of chunks, and per sequence. */
kvq_status kvq_decode_workspace_bytes(const kvq_store* k_store, const kvq_store* v_store,
                                      int batch, int num_q_heads, int max_len_hint,
                                      const kvq_decode_opts* opts, size_t* bytes);

/* Where `p` points, for callers deciding whether a buffer may be handed to a kernel:
 * *kind = 0 for device (or managed) memory, 1 for page-locked host memory mapped into the
 * current device's address space at the same address (usable in place where a call
 * allows host buffers), -1 otherwise (pageable host memory, unknown addresses).  A host
 * call (cudaPointerGetAttributes); KVQ_ERR_INVALID_ARG for null arguments. */
kvq_status kvq_pointer_kind(const void* p, int32_t* kind);

/* Zero a decode workspace (its arrival counters must be zero before its first use;
 * every completed kvq_flash_decode leaves them zero again).  Enqueued on `stream`.
 * Source: the split-K partials of rMLX issue #292 (see kvq_decode_workspace_bytes); the
 * counters are how the last CTA of a split finds out it is last.  workspace: device
 * memory, caller-owned.  KVQ_ERR_INVALID_ARG for a null pointer or zero size. */
kvq_status kvq_decode_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Split-K flash-decode over the quantized store (a2..a8):
 *   q          device bf16 [batch][num_q_heads][head_dim]
 *   k_store, v_store: same num_kv_heads, head_dim, page_size; codecs == `codec`.
 *   seq_lens   device int32 [batch], each in [0, max_len_hint]
 *   page_table device int32 [batch][max_pages]
 *   out        device fp32 [batch][num_q_heads][head_dim]
 *   Query head h reads KV head h / (num_q_heads / num_kv_heads); up to 16 query heads per
 *   KV head (32 for q8_0 K and V at head_dim 128 or 256 on the tensor-core kernel).
 *   softmax_scale <= 0 selects 1/sqrt(head_dim).
 *   max_len_hint: host-side upper bound of seq_lens, used to size the split without a
 *   device round trip; a longer sequence is truncated and recorded as a device fault.
 *   workspace: device memory of at least kvq_decode_workspace_bytes bytes, 16-byte
 *   aligned, zeroed once before its first use (kvq_decode_workspace_init); calls that
 *   share a workspace must not overlap on the device.
 * A sequence of length 0 yields zeros. */
kvq_status kvq_flash_decode(const void* q, const kvq_store* k_store, const kvq_store* v_store,
                            const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                            kvq_codec codec, float* out, int batch, int num_q_heads,
                            float softmax_scale, int max_len_hint,
                            const kvq_decode_opts* opts, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Decode of several query tokens per sequence against the same cache (speculative-draft
 * verification: halobench record clm-0022's shipped configuration drafts several tokens
 * per step, its --spec-draft-n-max note): the last num_tokens positions of each sequence are the
 * drafts, and query token i attends to positions [0, seq_lens[b] - num_tokens + i]
 * (causal among the drafts).  Every KV tile is read once for all of them.
 *   q    device bf16 [batch][num_q_heads][num_tokens][head_dim]
 *   out  device fp32 [batch][num_q_heads][num_tokens][head_dim]
 *   seq_lens[b] >= num_tokens (it counts the drafts, already appended with kvq_append_kv).
 * The workspace must hold kvq_decode_workspace_bytes(..., num_q_heads * num_tokens, ...).
 * Needs (num_q_heads / num_kv_heads) * num_tokens <= 16 (<= 32 for q8_0 K and V at
 * head_dim 128 or 256) and the tensor-core kernel (opts->variant 0 or 2), else
 * KVQ_ERR_UNSUPPORTED.  num_tokens == 1 is kvq_flash_decode.
 * A sequence shorter than num_tokens attends as if its drafts started at position 0
 * (query i sees positions below i + 1 - num_tokens + seq_lens[b], none if that is <= 0,
 * giving zeros). */
kvq_status kvq_flash_decode_multi(const void* q, const kvq_store* k_store, const kvq_store* v_store,
                                  const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                                  kvq_codec codec, float* out, int batch, int num_q_heads,
                                  int num_tokens, float softmax_scale, int max_len_hint,
                                  const kvq_decode_opts* opts, void* workspace,
                                  size_t workspace_bytes, void* stream);

/* Chunked prefill attention over the store (prompt processing: the pp512-at-depth arm of
 * halobench record clm-0022's tables, where dequantize-on-load also moved q8_0 prefill):
 * the last num_tokens positions of each sequence (already appended, e.g. with
 * kvq_append_kv) are the chunk's tokens, and token i attends to positions
 * [0, seq_lens[b] - num_tokens + i] (causal inside the chunk, everything before it).
 *   q    device bf16 [batch][num_tokens][num_q_heads][head_dim] (16-byte aligned)
 *   out  device fp32 [batch][num_tokens][num_q_heads][head_dim]
 * One launch, no workspace; each CTA streams the KV prefix of one KV head once.  Built for
 * the pairs of kvq_flash_decode's tensor-core kernel (bf16/bf16, f16/f16, q8_0/bf16,
 * q8_0/q8_0, q4s/q4s, q8_0/q4s, q4s/q8_0, q4s/bf16) at head_dim 64, 128 and 256, and for
 * q8_0/f16 and f16/q8_0 at 128.  At head_dim 128 a CTA owns 128 (token, head) query rows on
 * the 5th-generation tensor cores (scores, P and O in tensor memory, quantized tiles turned
 * once per CTA into exact f16 hi + lo operands); at 64 and 256, 64 rows on the warp-level
 * MMA path.  Other pairs give KVQ_ERR_UNSUPPORTED.  Unless K is bf16,
 * Q must lie in the f16 range (it is rounded to f16 once).  softmax_scale <= 0 selects
 * 1/sqrt(head_dim).  Device faults as for kvq_flash_decode. */
kvq_status kvq_prefill_attention(const void* q, const kvq_store* k_store, const kvq_store* v_store,
                                 const int32_t* seq_lens, const int32_t* page_table, int max_pages,
                                 kvq_codec codec, float* out, int batch, int num_q_heads,
                                 int num_tokens, float softmax_scale, void* stream);

/* One decode step with the append fused in (a1 followed by a2..a8, one launch of the
 * tensor-core kernel; the on-device append of rMLX issue #295 "Fix direction" done by
 * the decode kernel itself).  For every sequence b:
 *   - k_new[b] and v_new[b] (device bf16 [batch][num_kv_heads][head_dim], contiguous)
 *     are encoded into k_store and v_store at position seq_lens[b], exactly as
 *     kvq_append would encode them;
 *   - q attends over the seq_lens[b] + 1 tokens the stores then hold;
 *   - with advance != 0, seq_lens[b] is set to seq_lens[b] + 1 on the device, by the
 *     last of the sequence's CTAs once every one of them has read the old value;
 *     with advance == 0 it is left unchanged.
 * Arguments otherwise as for kvq_flash_decode, with seq_lens[b] + 1 <= max_len_hint.
 * The result equals kvq_append_kv(n_new = 1, advance) followed by kvq_flash_decode.
 * Only the tensor-core kernel implements it: opts->variant 1 gives KVQ_ERR_UNSUPPORTED.
 * A sequence whose new length does not fit gets no append and no advance and is
 * recorded as a device fault (KVQ_DEVICE_BAD_SEQ_LEN); a bad page of the new token is
 * recorded as KVQ_DEVICE_BAD_PAGE.
 * q, k_new, v_new and out may instead point to page-locked host memory that is mapped
 * into the device's address space (cudaHostAlloc, or a registered and mapped range; with
 * unified addressing the host address itself): the kernel then reads the step's inputs
 * and writes its output across the host link in place, so one call is the whole step
 * including its transfers.  The library does not check where these four pointers point;
 * any other host memory is undefined behaviour (as is an invalid device pointer).
 * seq_lens, page_table, the stores and the workspace stay in device memory. */
kvq_status kvq_flash_decode_append(const void* q, const void* k_new, const void* v_new,
                                   kvq_store* k_store, kvq_store* v_store, int32_t* seq_lens,
                                   const int32_t* page_table, int max_pages, kvq_codec codec,
                                   float* out, int batch, int num_q_heads, float softmax_scale,
                                   int max_len_hint, int advance, const kvq_decode_opts* opts,
                                   void* workspace, size_t workspace_bytes, void* stream);

/* kvq_flash_decode without a workspace argument, for callers that cannot allocate
 * device memory where they decode (inside host callbacks, under a memory manager that
 * owns all device memory, or in loops where cudaMalloc's implicit synchronization is
 * not acceptable).  The pages this library follows have no counterpart of this call.
 * The workspace is a fixed 16 MiB array in the library's own device memory (one per
 * GPU that loads the library, held until the process exits).  A call whose
 * kvq_decode_workspace_bytes would exceed 16 MiB returns KVQ_ERR_WORKSPACE and enqueues
 * nothing.  The first call on a device looks up the array's address (set-up, a
 * synchronous runtime query); make that first call before any stream capture.  Every
 * call zeroes the array's merge counters with an asynchronous memset on `stream`
 * (no allocation), after every argument check has passed: a call that fails a check
 * returns its error and enqueues nothing.  All calls share the one array, so calls that overlap on the device
 * (other streams, concurrent graphs) race; serialize them.  Other arguments, results
 * and errors are those of kvq_flash_decode. */
kvq_status kvq_flash_decode_static_ws(const void* q, const kvq_store* k_store,
                                      const kvq_store* v_store, const int32_t* seq_lens,
                                      const int32_t* page_table, int max_pages, kvq_codec codec,
                                      float* out, int batch, int num_q_heads,
                                      float softmax_scale, int max_len_hint,
                                      const kvq_decode_opts* opts, void* stream);

/* Wait for the device, read and clear the store's status word.  *device_code receives
 * the first recorded fault (KVQ_DEVICE_*), or 0.  Returns KVQ_ERR_DEVICE_FAULT when a
 * fault was recorded, KVQ_OK otherwise.  The only call that synchronizes.  The pages have
 * no counterpart: it is how kernels that never trap report bad device data. */
kvq_status kvq_store_get_error(kvq_store* store, int32_t* device_code);

/* Number of kernels (decode, append, combine, prefill, dequantize) this library has launched in this process
 * (a dispatch counter for benchmarks and tests: the pages prove their kernels ran by
 * counting dispatches, rMLX issue #295 "Finding" table and rMLX issue #292 "Symptom"). */
uint64_t kvq_launch_count(void);

/* Fault injection for tests of the device-timeout path (plumbing; the pages have no
 * counterpart: bounded waits are how this library's kernels avoid hanging on a stage that
 * never fills).  Applies to the tensor-core decode launches that follow in this process,
 * until reset with (0, -1):
 *   wait_limit  tries of each bounded mbarrier wait before it gives up (0 = the default,
 *               about four million);
 *   skip_tile   a tile of the first pipeline of every (sequence, KV head) unit that is
 *               never issued (neither its copies nor an arrival), or -1 for none.
 * With a tile skipped, that pipeline's waits run out: the kernel records
 * KVQ_DEVICE_TIMEOUT in the K store's status word and the call's output is invalid.  No
 * copy is left in flight (the skipped stage has none; every issued one is waited for
 * before the CTA exits), so the next call runs normally.  Process-wide, not synchronized
 * with launches from other threads.  KVQ_ERR_INVALID_ARG for wait_limit < 0 or
 * skip_tile < -1. */
kvq_status kvq_set_fault_injection(int32_t wait_limit, int32_t skip_tile);

/* Static string naming a status code (plumbing; the pages have no counterpart).  Never
 * NULL: unknown codes give "KVQ_UNKNOWN_STATUS". */
const char* kvq_status_string(kvq_status status);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */
