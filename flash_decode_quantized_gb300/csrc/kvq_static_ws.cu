// kvq_flash_decode_static_ws: the decode entry point for callers that must not allocate.
//
// kvq_flash_decode takes a caller-allocated workspace (split-K partials and merge
// counters).  Some callers cannot allocate device memory at the point where they
// decode: code running inside a CUDA host callback (which may make no CUDA call that
// allocates), engines whose memory manager owns all device memory and forbids
// allocations after start-up, and latency-critical loops where cudaMalloc's implicit
// device synchronization would stall the pipeline.  This entry point takes no
// workspace; it uses one fixed array in device memory that is part of the library image
// itself, so every GPU that loads the library holds that array until the process exits.
#include <mutex>

#include "kvq_internal.cuh"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(16) << 20;   // 16 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
kvq_status static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return KVQ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return KVQ_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return KVQ_OK;
}

}  // namespace

extern "C" kvq_status kvq_flash_decode_static_ws(const void* q, const kvq_store* k_store,
                                                 const kvq_store* v_store, const int32_t* seq_lens,
                                                 const int32_t* page_table, int max_pages, kvq_codec codec,
                                                 float* out, int batch, int num_q_heads, float softmax_scale,
                                                 int max_len_hint, const kvq_decode_opts* opts, void* stream) {
  if (!q || !k_store || !v_store || !seq_lens || !page_table || !out) return KVQ_ERR_INVALID_ARG;
  size_t need = 0, counters_off = 0;
  kvq_status st = kvq::decode_workspace_layout(k_store, v_store, batch, num_q_heads, max_len_hint, opts,
                                               &need, &counters_off);
  (void)counters_off;
  if (st != KVQ_OK) return st;
  if (need > kStaticWorkspaceBytes) return KVQ_ERR_WORKSPACE;
  void* ws = nullptr;
  st = static_workspace(&ws);
  if (st != KVQ_OK) return st;
  // The array keeps the previous call's contents: the merge counters this call relies on
  // are zeroed on `stream` right before the launch, after every argument check (a rejected
  // call enqueues nothing); the partials are fully written before they are read.
  return kvq::decode_reset(q, k_store, v_store, seq_lens, page_table, max_pages, codec, out, batch,
                           num_q_heads, softmax_scale, max_len_hint, opts, ws, kStaticWorkspaceBytes, stream);
}
