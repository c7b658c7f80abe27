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
// Set-up: the first call in a CUDA context, with that context's device
// current, asks the runtime for the array's device address
// (cudaGetSymbolAddress) and caches it under the context's unique id; a call
// from another context (a driver-API context of the host application, or the
// primary context recreated after cudaDeviceReset) looks the address up again
// in that context.  Make the first call of a context before any stream
// capture.  The host-side name of a __device__ array is only a stand-in, never
// a device address, so host code never passes it to a kernel.
//
// Every call shares the array and it keeps the last call's contents.  The
// decode kernels need none of it to start at zero (every slot they read was
// written earlier in the same call), so nothing is cleared.  Calls that
// overlap on the GPU (different streams, or graphs replayed concurrently)
// race on the array: serialise them.
#include "context_cache.h"
#include "pa_internal.h"

namespace pa {
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_NOALLOC_SCRATCH_BYTES];

ContextCache<void *> g_scratch_address;

// Device address of g_decode_scratch in the current context (looked up once per context).
pa_status scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return PA_ERR_CUDA;
  unsigned long long ctx = 0;
  pa_status st = current_context_id(&ctx);
  if (st != PA_OK) return st;
  void *ptr = nullptr;
  if (!g_scratch_address.get(dev, ctx,
                             [](void **v) { return cudaGetSymbolAddress(v, g_decode_scratch) == cudaSuccess && *v; },
                             &ptr))
    return dev < 0 || dev >= 64 ? PA_ERR_UNSUPPORTED : PA_ERR_CUDA;
  *out = ptr;
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_paged_attn_decode_noalloc(const void *q, const pa_kv_pool *pool,
                                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                  const int32_t *context_lens, int32_t num_seqs,
                                                  int32_t num_q_heads, int32_t max_context_len, float scale,
                                                  void *out, pa_stream_t stream) {
  // the same checks, in the same order, as pa_paged_attn_decode before its workspace
  pa_status st = pa::decode_check_args(q, pool, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                       num_q_heads, max_context_len, scale, out);
  if (st != PA_OK || num_seqs == 0) return st;
  const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, pool->num_kv_heads, max_context_len);
  if (need == 0) return PA_ERR_SHAPE;
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;  // beyond the fixed array
  void *scratch = nullptr;
  st = pa::scratch_address(&scratch);
  if (st != PA_OK) return st;
  return pa_paged_attn_decode(q, pool, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                              max_context_len, scale, out, scratch, (size_t)PA_NOALLOC_SCRATCH_BYTES, stream);
}
