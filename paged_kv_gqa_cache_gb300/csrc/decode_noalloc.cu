// pa_paged_attn_decode_noalloc: paged decode attention that allocates nothing.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: a
// plugin running inside a host application that owns all device memory, or a
// serving step that is not allowed to allocate at all.  This entry point
// computes exactly what pa_paged_attn_decode computes, but its split-K
// scratch lives in one fixed array compiled into the library.  Each GPU that
// loads the library holds that array (PA_NOALLOC_SCRATCH_BYTES) until the
// process exits.
//
// Set-up: the first call on a device, with that device current, asks the
// runtime for the array's device address (cudaGetSymbolAddress) and caches
// it; make that first call before any stream capture.  The host-side name of
// a __device__ array is only a stand-in, never a device address, so host code
// never passes it to a kernel.
//
// Every call shares the array and it keeps the last call's contents.  The
// decode kernels need none of it to start at zero (every slot they read was
// written earlier in the same call), so nothing is cleared.  Calls that
// overlap on the GPU (different streams, or graphs replayed concurrently)
// race on the array: serialise them.
#include <mutex>

#include "pa_internal.h"

namespace pa {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (set up once per device).
pa_status scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess || !ptr) return PA_ERR_CUDA;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_paged_attn_decode_noalloc(const void *q, const pa_kv_pool *pool,
                                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                  const int32_t *context_lens, int32_t num_seqs,
                                                  int32_t num_q_heads, int32_t max_context_len, float scale,
                                                  void *out, pa_stream_t stream) {
  if (!pool) return PA_ERR_NULL;
  if (num_seqs < 0) return PA_ERR_SHAPE;
  if (num_seqs == 0) return PA_OK;
  const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, pool->num_kv_heads, max_context_len);
  if (need == 0) return PA_ERR_SHAPE;
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;  // beyond the fixed array
  void *scratch = nullptr;
  const pa_status st = pa::scratch_address(&scratch);
  if (st != PA_OK) return st;
  return pa_paged_attn_decode(q, pool, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                              max_context_len, scale, out, scratch, (size_t)PA_NOALLOC_SCRATCH_BYTES, stream);
}
