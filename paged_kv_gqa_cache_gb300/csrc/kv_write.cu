// kv_cache_write for sm_103a: scatter the K/V rows of the step's new tokens
// into their pool slots (page "Модуль 12: Финальный проект: мини-движок
// инференса", qwen_serve/paged.py, PagedKVCache.write).
//
// A pure bit copy, bound by HBM bandwidth: each token row (num_kv_heads x 128
// 16-bit values, 2 KB for 8 KV heads) is read once from k/v and written once
// into slot slot_mapping[t] of the pool, with 128-bit coalesced loads and
// stores.  Consecutive threads take consecutive 16-byte vectors of one row, so
// every warp moves whole 512-byte runs.
#include "pa_device.cuh"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) kv_write_kernel(const WriteParams p) {
  griddep_wait();
  // the next kernel may start its set-up now; it still waits for this grid to
  // complete before it reads anything (griddep_wait)
  griddep_launch_dependents();
  const int64_t total = (int64_t)p.num_tokens * p.row_vecs;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int t = (int)(i / p.row_vecs);
    const int vi = (int)(i - (int64_t)t * p.row_vecs);
    const int64_t slot = __ldg(p.slots + t);
    if (slot < 0 || slot >= p.num_slots) {
      if (vi == 0) set_error(p.err, PA_ERR_RANGE, t);
      continue;
    }
    const uint4 kv = ld_nc_v4(static_cast<const uint4 *>(p.k) + i);
    const uint4 vv = ld_nc_v4(static_cast<const uint4 *>(p.v) + i);
    st_v4(static_cast<uint4 *>(p.k_cache) + slot * p.row_vecs + vi, kv);
    st_v4(static_cast<uint4 *>(p.v_cache) + slot * p.row_vecs + vi, vv);
  }
}

}  // namespace

cudaError_t launch_kv_write(const WriteParams &p, cudaStream_t stream) {
  const int64_t total = (int64_t)p.num_tokens * p.row_vecs;
  int64_t grid = (total + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_pdl(kv_write_kernel, dim3((unsigned)grid), dim3(256), 0, stream, p);
}

}  // namespace pa
