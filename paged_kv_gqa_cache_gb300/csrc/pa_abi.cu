// The C-ABI of libpagedattn: argument validation, per-device state (SM count,
// error word), TMA tensor-map encoding, and dispatch to the kernels.  Every
// check that can be made on the host is made here, before anything is
// enqueued; see include/pagedattn.h for the contract of each call.
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>
#include <mutex>

#include "context_cache.h"
#include "pa_internal.h"

namespace pa {

// err[0]: first status recorded by a kernel on this device, err[1]: its detail.
__device__ int g_error_word[2];

namespace {

thread_local int t_last_cuda_error = 0;
thread_local unsigned long long t_context_id = 0;

struct DeviceState {
  bool ready = false;
  int sm_count = 0;
  int *err = nullptr;
};

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
int g_sm_count[kMaxDevices] = {};        // per device, whatever the context
thread_local DeviceState t_state;        // this thread's current device and context
ContextCache<int *, kMaxDevices> g_error_word_address;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;

pa_status cuda_fail(cudaError_t e) {
  t_last_cuda_error = (int)e;
  return PA_ERR_CUDA;
}

// Driver entry points the library calls directly (resolved once).
std::atomic<bool> g_entry_points_ready{false};
pa_status driver_entry_points() {
  if (g_entry_points_ready.load(std::memory_order_acquire)) return PA_OK;
  std::lock_guard<std::mutex> lock(g_mutex);
  struct Want {
    const char *name;
    void **fn;
    int version;
  } want[] = {{"cuTensorMapEncodeTiled", reinterpret_cast<void **>(&g_encode), 12000},
              {"cuCtxGetCurrent", reinterpret_cast<void **>(&g_ctx_get_current), 4000},
              {"cuCtxGetId", reinterpret_cast<void **>(&g_ctx_get_id), 12000}};
  for (const Want &w : want) {
    if (*w.fn) continue;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion(w.name, &fn, w.version, cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_fail(e);
    if (q != cudaDriverEntryPointSuccess || !fn) return PA_ERR_CUDA;
    *w.fn = fn;
  }
  g_entry_points_ready.store(true, std::memory_order_release);
  return PA_OK;
}

}  // namespace

// The unique id of the current CUDA context.  With no context current, the
// current device's primary context is initialised and made current first
// (what the runtime would do on the next kernel launch).
pa_status current_context_id(unsigned long long *id) {
  pa_status st = driver_entry_points();
  if (st != PA_OK) return st;
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return PA_ERR_CUDA;
  if (!ctx) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);  // initialises the device's primary context
    if (e != cudaSuccess) return cuda_fail(e);
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return PA_ERR_CUDA;
  }
  unsigned long long v = 0;
  if (g_ctx_get_id(ctx, &v) != CUDA_SUCCESS || v == 0) return PA_ERR_CUDA;
  *id = v;
  return PA_OK;
}

unsigned long long launch_context_id() { return t_context_id; }

namespace {

// Set-up per device (SM count) and per context (the error word's address),
// with that device current.  Every entry point that launches calls it first,
// which also records the context for launch_context_id().
pa_status device_state(DeviceState **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  unsigned long long ctx = 0;
  pa_status st = current_context_id(&ctx);
  if (st != PA_OK) return st;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_sm_count[dev] == 0) {
      e = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    sms = g_sm_count[dev];
  }
  // The host-side name of a __device__ variable is not a device address;
  // ask the runtime for the real one, in this context.
  int *err = nullptr;
  cudaError_t fetch_err = cudaSuccess;
  if (!g_error_word_address.get(dev, ctx,
                                [&](int **v) {
                                  fetch_err = cudaGetSymbolAddress(reinterpret_cast<void **>(v), g_error_word);
                                  return fetch_err == cudaSuccess && *v != nullptr;
                                },
                                &err))
    return fetch_err != cudaSuccess ? cuda_fail(fetch_err) : PA_ERR_CUDA;
  t_state.ready = true;
  t_state.sm_count = sms;
  t_state.err = err;
  t_context_id = ctx;
  *out = &t_state;
  return PA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

pa_status check_pool(const pa_kv_pool *pool) {
  if (!pool || !pool->k_cache || !pool->v_cache) return PA_ERR_NULL;
  if (pool->dtype != PA_F16 && pool->dtype != PA_BF16) return PA_ERR_DTYPE;
  if (pool->block_size != kBlock || pool->head_dim != kHeadDim) return PA_ERR_UNSUPPORTED;
  if (pool->num_blocks < 1 || pool->num_kv_heads < 1 || pool->num_kv_heads > 256) return PA_ERR_SHAPE;
  if (!aligned16(pool->k_cache) || !aligned16(pool->v_cache)) return PA_ERR_ALIGN;
  return PA_OK;
}

pa_status check_group(int num_q_heads, int num_kv_heads, int *group) {
  if (num_q_heads < 1 || num_q_heads % num_kv_heads != 0) return PA_ERR_SHAPE;
  const int g = num_q_heads / num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PA_ERR_UNSUPPORTED;
  *group = g;
  return PA_OK;
}

CUtensorMapDataType map_dtype(int dtype) {
  return dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// The pool as a 4-D tensor {dim, kv head, in-block slot, block}.  The prefill
// kernel feeds tensor cores and needs the 128-byte swizzled layout, so its
// boxes are {64 dims, 1 head, 16 slots, 1 block} (half a page of one KV head,
// 2 KB); the decode kernel reads with CUDA cores and takes a whole page of one
// KV head per box, {128, 1, 16, 1} unswizzled (4 KB).
bool pool_map(CUtensorMap *map, const pa_kv_pool *pool, void *base, bool whole_page_box) {
  const uint64_t hkv = (uint64_t)pool->num_kv_heads;
  const uint64_t dims[4] = {(uint64_t)kHeadDim, hkv, (uint64_t)kBlock, (uint64_t)pool->num_blocks};
  const uint64_t strides[3] = {kHeadDim * 2ull, hkv * kHeadDim * 2ull, kBlock * hkv * kHeadDim * 2ull};
  const uint32_t box[4] = {whole_page_box ? 128u : 64u, 1, (uint32_t)kBlock, 1};
  return encode_tensor_map(map, map_dtype(pool->dtype), 4, base, dims, strides, box,
                           whole_page_box ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B);
}

// The pool's V for the prefill: one box per page of one KV head with both
// 64-dim halves, as the 5-D tensor {64 dims, 16 slots, 2 halves, kv head,
// block} (strides: slot Hkv * 256 B, half 128 B, head 256 B, block 16 * Hkv *
// 256 B).  The box {64, 16, 2, 1, 1} lands in shared memory as the 16 rows of
// dims 0..63 (2 KB) followed by the 16 rows of dims 64..127, 128-byte
// swizzled: the MN-major layout the P V product reads with the two halves
// 2 KB apart.  A key tile then takes 8 boxes of 4 KB instead of 16 of 2 KB.
bool pool_map_vpages(CUtensorMap *map, const pa_kv_pool *pool, void *base) {
  const uint64_t hkv = (uint64_t)pool->num_kv_heads;
  const uint64_t dims[5] = {64, (uint64_t)kBlock, 2, hkv, (uint64_t)pool->num_blocks};
  const uint64_t strides[4] = {hkv * kHeadDim * 2ull, 128ull, kHeadDim * 2ull, kBlock * hkv * kHeadDim * 2ull};
  const uint32_t box[5] = {64u, (uint32_t)kBlock, 2u, 1u, 1u};
  return encode_tensor_map(map, map_dtype(pool->dtype), 5, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

// int8 pool [P2 section 5]: codes as a 4-D tensor of bytes {dim, kv head,
// slot, block}; the decode takes one page of one KV head per box (2 KB).
pa_status check_pool_q8(const pa_kv_pool_q8 *pool) {
  if (!pool || !pool->k_cache || !pool->v_cache || !pool->k_scale || !pool->v_scale) return PA_ERR_NULL;
  if (pool->block_size != kBlock || pool->head_dim != kHeadDim) return PA_ERR_UNSUPPORTED;
  if (pool->num_blocks < 1 || pool->num_kv_heads < 1 || pool->num_kv_heads > 256) return PA_ERR_SHAPE;
  if (!aligned16(pool->k_cache) || !aligned16(pool->v_cache) || !aligned16(pool->k_scale) ||
      !aligned16(pool->v_scale))
    return PA_ERR_ALIGN;
  return PA_OK;
}

bool pool_map_q8(CUtensorMap *map, const pa_kv_pool_q8 *pool, void *base) {
  const uint64_t hkv = (uint64_t)pool->num_kv_heads;
  const uint64_t dims[4] = {(uint64_t)kHeadDim, hkv, (uint64_t)kBlock, (uint64_t)pool->num_blocks};
  const uint64_t strides[3] = {kHeadDim * 1ull, hkv * kHeadDim, kBlock * hkv * kHeadDim};
  const uint32_t box[4] = {128u, 1, (uint32_t)kBlock, 1};
  // a page row of one KV head is 128 bytes here, 1 KB apart (8 heads): promoting
  // each fetch to 256 bytes would pull in another head's row
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, base, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

// The decode call on a 16-bit pool (pool16) or an int8 pool (pool8), after the
// pool's own checks: every other argument is checked before any CUDA call.
pa_status decode_call(const void *q, int dtype, const pa_kv_pool *pool16, const pa_kv_pool_q8 *pool8,
                      const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                      int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len, float scale, int32_t window,
                      void *out, void *workspace, size_t workspace_bytes, cudaStream_t stream,
                      const void *k_new = nullptr, const void *v_new = nullptr, bool f8 = false,
                      uint32_t flags = 0) {
  const bool q8 = pool8 != nullptr;
  const int num_kv_heads = q8 ? pool8->num_kv_heads : pool16->num_kv_heads;
  const int num_blocks = q8 ? pool8->num_blocks : pool16->num_blocks;
  if (num_seqs < 0) return PA_ERR_SHAPE;
  if (num_seqs == 0) return PA_OK;
  if (!q || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  if (!workspace) return PA_ERR_WORKSPACE;
  int group = 0;
  pa_status st = check_group(num_q_heads, num_kv_heads, &group);
  if (st != PA_OK) return st;
  if (max_blocks_per_seq < 1 || max_context_len < 1 ||
      (int64_t)max_context_len > (int64_t)max_blocks_per_seq * kBlock)
    return PA_ERR_SHAPE;
  if (num_seqs > 16384) return PA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_SHAPE;
  if (window < 0) return PA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(out) || !aligned16(workspace) || !aligned4(block_tables) ||
      !aligned4(context_lens) || !aligned16(k_new) || !aligned16(v_new))
    return PA_ERR_ALIGN;
  if (workspace_bytes < decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads)) return PA_ERR_WORKSPACE;
  DeviceState *d = nullptr;
  if ((st = device_state(&d)) != PA_OK) return st;  // also readies the tensor-map encoder
  CUtensorMap kmap, vmap;
  const bool maps = q8 ? pool_map_q8(&kmap, pool8, pool8->k_cache) && pool_map_q8(&vmap, pool8, pool8->v_cache)
                       : pool_map(&kmap, pool16, pool16->k_cache, true) &&
                             pool_map(&vmap, pool16, pool16->v_cache, true);
  if (!maps) return PA_ERR_CUDA;

  DecodeParams p{};
  if (!decode_workspace_carve(workspace, workspace_bytes, num_seqs, num_q_heads, num_kv_heads, p))
    return PA_ERR_WORKSPACE;
  p.q = q;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.err = d->err;
  p.k_scale = q8 ? pool8->k_scale : nullptr;
  p.v_scale = q8 ? pool8->v_scale : nullptr;
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_pool = q8 ? nullptr : pool16->k_cache;
  p.v_pool = q8 ? nullptr : pool16->v_cache;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.num_kv_heads = num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.num_blocks = num_blocks;
  p.window = window;
  p.early_pages = (flags & PA_DECODE_EARLY_PAGES) ? 1 : 0;
  // a workspace whose counters the caller keeps zero: one launch over all SMs, split items merged in it
  p.counters = (flags & PA_DECODE_ZEROED_WORKSPACE)
                   ? reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) +
                                                 decode_workspace_counters_offset(num_seqs, num_q_heads, num_kv_heads))
                   : nullptr;
  p.scale_log2 = scale * 1.4426950408889634f;

  // Upper bound on the pages of one item (a window of W keys spans at most
  // (W - 1) / 16 + 2 pages) and of the call; aim for at least 4 pages per warp.
  int item_pages = (max_context_len + kBlock - 1) / kBlock;
  if (window > 0 && (window - 1) / kBlock + 2 < item_pages) item_pages = (window - 1) / kBlock + 2;
  const int64_t pages_hint = (int64_t)num_seqs * num_kv_heads * item_pages;
  // one launch with the merge inside: as many warps as fit (every page in flight early); else aim for
  // at least 4 pages per warp
  int64_t workers = p.counters ? (pages_hint + 1) / 2 : (pages_hint + 3) / 4;
  if (workers > kDecodeMaxWorkers) workers = kDecodeMaxWorkers;
  cudaError_t e = launch_decode(p, kmap, vmap, dtype, group, (int)workers, item_pages, q8, q8 && f8, stream);
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // namespace

// The checks pa_paged_attn_decode makes before it looks at its workspace, in
// the same order, for the allocation-free entry point (which has none).
pa_status decode_check_args(const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t max_context_len, float scale, void *out) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  if (num_seqs < 0) return PA_ERR_SHAPE;
  if (num_seqs == 0) return PA_OK;
  if (!q || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  int group = 0;
  if ((st = check_group(num_q_heads, pool->num_kv_heads, &group)) != PA_OK) return st;
  if (max_blocks_per_seq < 1 || max_context_len < 1 ||
      (int64_t)max_context_len > (int64_t)max_blocks_per_seq * kBlock)
    return PA_ERR_SHAPE;
  if (num_seqs > 16384) return PA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(out) || !aligned4(block_tables) || !aligned4(context_lens)) return PA_ERR_ALIGN;
  return PA_OK;
}

int sm_count() {
  DeviceState *d = nullptr;
  if (device_state(&d) != PA_OK) return 1;
  return d->sm_count;
}

bool encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, int rank, void *base,
                       const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                       CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promotion) {
  if (!g_encode) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, dtype, (cuuint32_t)rank, base, reinterpret_cast<const cuuint64_t *>(dims),
                        reinterpret_cast<const cuuint64_t *>(strides_bytes),
                        reinterpret_cast<const cuuint32_t *>(box), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle, promotion, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace pa

using namespace pa;

extern "C" {

int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

int32_t pa_last_cuda_error(void) { return t_last_cuda_error; }

const char *pa_status_string(int32_t status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: a size is negative, inconsistent or over a limit";
    case PA_ERR_DTYPE: return "PA_ERR_DTYPE: dtype must be PA_F16 or PA_BF16";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: head_dim 128, block 16 and head ratio 1/2/4/8 only";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA call failed";
    case PA_ERR_RANGE: return "PA_ERR_RANGE: block id, slot or length out of range";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: a bounded wait gave up";
    case PA_ERR_ALIGN: return "PA_ERR_ALIGN: a pointer is not 16-byte aligned";
    case PA_ERR_NO_BLOCKS: return "PA_ERR_NO_BLOCKS: not enough free blocks";
    case PA_ERR_STATE: return "PA_ERR_STATE: allocator call out of order";
    default: return "unknown pa_status";
  }
}

pa_status pa_kv_cache_write(const void *k, const void *v, const int64_t *slot_mapping, int32_t num_tokens,
                            const pa_kv_pool *pool, pa_stream_t stream) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping) return PA_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)) return PA_ERR_ALIGN;
  DeviceState *d = nullptr;
  if ((st = device_state(&d)) != PA_OK) return st;
  WriteParams p;
  p.k = k;
  p.v = v;
  p.slots = slot_mapping;
  p.k_cache = pool->k_cache;
  p.v_cache = pool->v_cache;
  p.num_slots = (int64_t)pool->num_blocks * kBlock;
  p.num_tokens = num_tokens;
  p.row_vecs = pool->num_kv_heads * kHeadDim * 2 / 16;
  p.err = d->err;
  cudaError_t e = launch_kv_write(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t max_context_len) {
  if (num_seqs < 0 || num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads != 0 ||
      max_context_len < 0)
    return 0;
  return decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads);
}

int32_t pa_decode_kernel_launches(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len) {
  if (num_seqs < 1 || num_seqs > 16384 || num_kv_heads < 1 || max_context_len < 1) return 0;
  if (sm_count() < 1) return 0;
  return decode_item_ctas(num_seqs * num_kv_heads, (max_context_len + kBlock - 1) / kBlock) > 0 ? 1 : 2;
}

pa_status pa_paged_attn_decode(const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                               int32_t num_q_heads, int32_t max_context_len, float scale, void *out,
                               void *workspace, size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  return decode_call(q, pool->dtype, pool, nullptr, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, max_context_len, scale, 0, out, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream));
}

pa_status pa_paged_attn_decode_append(const void *q, const void *k_new, const void *v_new, const pa_kv_pool *pool,
                                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                                      const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                      int32_t max_context_len, float scale, void *out, void *workspace,
                                      size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  if (num_seqs > 0 && (!k_new || !v_new)) return PA_ERR_NULL;
  return decode_call(q, pool->dtype, pool, nullptr, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, max_context_len, scale, 0, out, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), k_new, v_new);
}

pa_status pa_paged_attn_decode_ex(const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                                  int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t max_context_len, float scale, int32_t window,
                                  const void *k_new, const void *v_new, uint32_t flags, void *out,
                                  void *workspace, size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  if ((k_new == nullptr) != (v_new == nullptr)) return PA_ERR_NULL;
  if (k_new && window != 0) return PA_ERR_UNSUPPORTED;
  if (flags & ~(uint32_t)(PA_DECODE_EARLY_PAGES | PA_DECODE_ZEROED_WORKSPACE)) return PA_ERR_UNSUPPORTED;
  return decode_call(q, pool->dtype, pool, nullptr, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, max_context_len, scale, window, out, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), k_new, v_new, false, flags);
}

pa_status pa_paged_attn_decode_window(const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t max_context_len, float scale, int32_t window,
                                      void *out, void *workspace, size_t workspace_bytes, pa_stream_t stream) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  return decode_call(q, pool->dtype, pool, nullptr, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, max_context_len, scale, window, out, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream));
}

namespace {

// The quantising write into an 8-bit pool: int8 codes, or E4M3 codes when f8.
pa_status write_8bit(const void *k, const void *v, int32_t dtype, const int64_t *slot_mapping, int32_t num_tokens,
                     const pa_kv_pool_q8 *pool, bool f8, pa_stream_t stream) {
  pa_status st = check_pool_q8(pool);
  if (st != PA_OK) return st;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (num_tokens < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping) return PA_ERR_NULL;
  if (!aligned16(k) || !aligned16(v) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)) return PA_ERR_ALIGN;
  DeviceState *d = nullptr;
  if ((st = device_state(&d)) != PA_OK) return st;
  WriteQ8Params p;
  p.k = k;
  p.v = v;
  p.slots = slot_mapping;
  p.k_cache = static_cast<int8_t *>(pool->k_cache);
  p.v_cache = static_cast<int8_t *>(pool->v_cache);
  p.k_scale = pool->k_scale;
  p.v_scale = pool->v_scale;
  p.num_slots = (int64_t)pool->num_blocks * kBlock;
  p.num_tokens = num_tokens;
  p.num_kv_heads = pool->num_kv_heads;
  p.err = d->err;
  cudaError_t e = launch_kv_write_q8(p, dtype, f8, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status decode_8bit(const void *q, int32_t dtype, const pa_kv_pool_q8 *pool, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                      int32_t num_q_heads, int32_t max_context_len, float scale, void *out, void *workspace,
                      size_t workspace_bytes, bool f8, pa_stream_t stream, uint32_t flags = 0) {
  pa_status st = check_pool_q8(pool);
  if (st != PA_OK) return st;
  if (dtype != PA_F16 && dtype != PA_BF16) return PA_ERR_DTYPE;
  return decode_call(q, dtype, nullptr, pool, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_q_heads, max_context_len, scale, 0, out, workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream), nullptr, nullptr, f8, flags);
}

}  // namespace

pa_status pa_kv_cache_write_q8(const void *k, const void *v, int32_t dtype, const int64_t *slot_mapping,
                               int32_t num_tokens, const pa_kv_pool_q8 *pool, pa_stream_t stream) {
  return write_8bit(k, v, dtype, slot_mapping, num_tokens, pool, false, stream);
}

pa_status pa_kv_cache_write_f8(const void *k, const void *v, int32_t dtype, const int64_t *slot_mapping,
                               int32_t num_tokens, const pa_kv_pool_q8 *pool, pa_stream_t stream) {
  return write_8bit(k, v, dtype, slot_mapping, num_tokens, pool, true, stream);
}

pa_status pa_paged_attn_decode_q8(const void *q, int32_t dtype, const pa_kv_pool_q8 *pool,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_context_len, float scale, void *out, void *workspace,
                                  size_t workspace_bytes, pa_stream_t stream) {
  return decode_8bit(q, dtype, pool, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                     max_context_len, scale, out, workspace, workspace_bytes, false, stream);
}

pa_status pa_paged_attn_decode_q8_ex(const void *q, int32_t dtype, const pa_kv_pool_q8 *pool, int32_t codes,
                                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                                     const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                     int32_t max_context_len, float scale, uint32_t flags, void *out,
                                     void *workspace, size_t workspace_bytes, pa_stream_t stream) {
  if (codes != PA_CODES_INT8 && codes != PA_CODES_E4M3) return PA_ERR_UNSUPPORTED;
  if (flags & ~(uint32_t)(PA_DECODE_EARLY_PAGES | PA_DECODE_ZEROED_WORKSPACE)) return PA_ERR_UNSUPPORTED;
  return decode_8bit(q, dtype, pool, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                     max_context_len, scale, out, workspace, workspace_bytes, codes == PA_CODES_E4M3, stream,
                     flags);
}

pa_status pa_paged_attn_decode_f8(const void *q, int32_t dtype, const pa_kv_pool_q8 *pool,
                                  const int32_t *block_tables, int32_t max_blocks_per_seq,
                                  const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_context_len, float scale, void *out, void *workspace,
                                  size_t workspace_bytes, pa_stream_t stream) {
  return decode_8bit(q, dtype, pool, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                     max_context_len, scale, out, workspace, workspace_bytes, true, stream);
}

namespace {

// The prefill call; with a workspace (and at most kMaxChunksBalanced chunks)
// the balanced launch runs, else the plain one.
// q (and out) as a 3-D tensor {dim, query head, token}; boxes of {64 dims,
// G heads, 128/G tokens} give 128 rows (token-major, head-minor) of 128 bytes.
bool query_maps(CUtensorMap *qmap, CUtensorMap *omap, const void *q, void *out, int dtype, int num_q_heads,
                int total_q_tokens, int group) {
  const uint64_t dims[3] = {(uint64_t)kHeadDim, (uint64_t)num_q_heads, (uint64_t)total_q_tokens};
  const uint64_t strides[2] = {kHeadDim * 2ull, (uint64_t)num_q_heads * kHeadDim * 2ull};
  const uint32_t box[3] = {64, (uint32_t)group, (uint32_t)(128 / group)};
  return encode_tensor_map(qmap, map_dtype(dtype), 3, const_cast<void *>(q), dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_tensor_map(omap, map_dtype(dtype), 3, out, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

pa_status prefill_call(const void *q, const int32_t *chunk_starts, const int32_t *chunk_lens, const pa_kv_pool *pool,
                       const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                       int32_t num_chunks, int32_t num_q_heads, int32_t total_q_tokens, int32_t max_chunk_len,
                       float scale, int32_t window, void *out, void *workspace, size_t workspace_bytes,
                       pa_stream_t stream) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  if (num_chunks < 0 || total_q_tokens < 0 || window < 0) return PA_ERR_SHAPE;
  if (num_chunks == 0) return PA_OK;
  if (!q || !chunk_starts || !chunk_lens || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  int group = 0;
  if ((st = check_group(num_q_heads, pool->num_kv_heads, &group)) != PA_OK) return st;
  if (max_chunk_len < 1 || max_chunk_len > PA_MAX_CHUNK_LEN || max_blocks_per_seq < 1) return PA_ERR_SHAPE;
  if (total_q_tokens < 1) return PA_ERR_SHAPE;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(out) || !aligned4(block_tables) || !aligned4(context_lens) ||
      !aligned4(chunk_starts) || !aligned4(chunk_lens))
    return PA_ERR_ALIGN;
  DeviceState *d = nullptr;
  if ((st = device_state(&d)) != PA_OK) return st;

  PrefillParams p{};
  p.q = q;
  p.k_cache = pool->k_cache;
  p.v_cache = pool->v_cache;
  p.chunk_starts = chunk_starts;
  p.chunk_lens = chunk_lens;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.err = d->err;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_chunks = num_chunks;
  p.num_kv_heads = pool->num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.num_blocks = pool->num_blocks;
  p.total_q_tokens = total_q_tokens;
  p.max_chunk_len = max_chunk_len;
  p.window = window;
  p.scale_log2 = scale * 1.4426950408889634f;

  CUtensorMap kmap, vmap, qmap, omap;
  if (!pool_map(&kmap, pool, pool->k_cache, false) || !pool_map_vpages(&vmap, pool, pool->v_cache) ||
      !query_maps(&qmap, &omap, q, out, pool->dtype, num_q_heads, total_q_tokens, group))
    return PA_ERR_CUDA;
  if (workspace && num_chunks <= kMaxChunksBalanced) {
    if (!aligned16(workspace)) return PA_ERR_ALIGN;
    if (!prefill_workspace_carve(workspace, workspace_bytes, num_chunks, num_q_heads, pool->num_kv_heads,
                                 max_chunk_len, d->sm_count, p))
      return PA_ERR_WORKSPACE;
  }
  cudaError_t e =
      launch_prefill(p, kmap, vmap, qmap, omap, pool->dtype, group, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // namespace

pa_status pa_paged_attn_prefill_chunk_q8(const void *q, int32_t dtype, const int32_t *chunk_starts,
                                         const int32_t *chunk_lens, const pa_kv_pool_q8 *pool, int32_t codes,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *context_lens, int32_t num_chunks, int32_t num_q_heads,
                                         int32_t total_q_tokens, int32_t max_chunk_len, float scale, void *out,
                                         pa_stream_t stream) {
  pa_status st = check_pool_q8(pool);
  if (st != PA_OK) return st;
  if (dtype != PA_BF16 && dtype != PA_F16) return PA_ERR_DTYPE;
  if (codes != PA_CODES_INT8 && codes != PA_CODES_E4M3) return PA_ERR_UNSUPPORTED;
  if (num_chunks < 0 || total_q_tokens < 0) return PA_ERR_SHAPE;
  if (num_chunks == 0) return PA_OK;
  if (!q || !chunk_starts || !chunk_lens || !block_tables || !context_lens || !out) return PA_ERR_NULL;
  int group = 0;
  if ((st = check_group(num_q_heads, pool->num_kv_heads, &group)) != PA_OK) return st;
  if (max_chunk_len < 1 || max_chunk_len > PA_MAX_CHUNK_LEN || max_blocks_per_seq < 1) return PA_ERR_SHAPE;
  if (total_q_tokens < 1) return PA_ERR_SHAPE;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(out) || !aligned4(block_tables) || !aligned4(context_lens) ||
      !aligned4(chunk_starts) || !aligned4(chunk_lens))
    return PA_ERR_ALIGN;
  DeviceState *d = nullptr;
  if ((st = device_state(&d)) != PA_OK) return st;  // also readies the tensor-map encoder
  CUtensorMap kmap, vmap, qmap, omap;
  if (!pool_map_q8(&kmap, pool, pool->k_cache) || !pool_map_q8(&vmap, pool, pool->v_cache) ||
      !query_maps(&qmap, &omap, q, out, dtype, num_q_heads, total_q_tokens, group))
    return PA_ERR_CUDA;
  PrefillParams p{};
  p.q = q;
  p.k_cache = pool->k_cache;
  p.v_cache = pool->v_cache;
  p.k_scale = pool->k_scale;
  p.v_scale = pool->v_scale;
  p.chunk_starts = chunk_starts;
  p.chunk_lens = chunk_lens;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.out = out;
  p.err = d->err;
  p.max_blocks_per_seq = max_blocks_per_seq;
  p.num_chunks = num_chunks;
  p.num_kv_heads = pool->num_kv_heads;
  p.num_q_heads = num_q_heads;
  p.num_blocks = pool->num_blocks;
  p.total_q_tokens = total_q_tokens;
  p.max_chunk_len = max_chunk_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaError_t e = launch_prefill8(p, kmap, vmap, qmap, omap, dtype, group, codes == PA_CODES_E4M3,
                                  static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t pa_prefill_workspace_bytes(int32_t num_chunks, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t max_chunk_len) {
  if (num_chunks < 1 || num_kv_heads < 1 || num_q_heads < 1 || num_q_heads % num_kv_heads != 0 ||
      max_chunk_len < 1 || max_chunk_len > PA_MAX_CHUNK_LEN)
    return 0;
  const int sms = sm_count();
  return prefill_workspace_bytes(num_chunks, num_q_heads, num_kv_heads, max_chunk_len, sms > 0 ? sms : 1);
}

pa_status pa_paged_attn_prefill_chunk_window(const void *q, const int32_t *chunk_starts,
                                             const int32_t *chunk_lens, const pa_kv_pool *pool,
                                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                                             const int32_t *context_lens, int32_t num_chunks, int32_t num_q_heads,
                                             int32_t total_q_tokens, int32_t max_chunk_len, float scale,
                                             int32_t window, void *out, pa_stream_t stream) {
  return prefill_call(q, chunk_starts, chunk_lens, pool, block_tables, max_blocks_per_seq, context_lens, num_chunks,
                      num_q_heads, total_q_tokens, max_chunk_len, scale, window, out, nullptr, 0, stream);
}

pa_status pa_paged_attn_prefill_chunk_ex(const void *q, const int32_t *chunk_starts, const int32_t *chunk_lens,
                                         const pa_kv_pool *pool, const int32_t *block_tables,
                                         int32_t max_blocks_per_seq, const int32_t *context_lens,
                                         int32_t num_chunks, int32_t num_q_heads, int32_t total_q_tokens,
                                         int32_t max_chunk_len, float scale, int32_t window, void *out,
                                         void *workspace, size_t workspace_bytes, pa_stream_t stream) {
  if (!workspace && num_chunks > 0) return PA_ERR_WORKSPACE;
  return prefill_call(q, chunk_starts, chunk_lens, pool, block_tables, max_blocks_per_seq, context_lens, num_chunks,
                      num_q_heads, total_q_tokens, max_chunk_len, scale, window, out, workspace, workspace_bytes,
                      stream);
}

pa_status pa_paged_attn_prefill_chunk(const void *q, const int32_t *chunk_starts, const int32_t *chunk_lens,
                                      const pa_kv_pool *pool, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      int32_t num_chunks, int32_t num_q_heads, int32_t total_q_tokens,
                                      int32_t max_chunk_len, float scale, void *out, pa_stream_t stream) {
  return pa_paged_attn_prefill_chunk_window(q, chunk_starts, chunk_lens, pool, block_tables, max_blocks_per_seq,
                                            context_lens, num_chunks, num_q_heads, total_q_tokens, max_chunk_len,
                                            scale, 0, out, stream);
}

pa_status pa_qk_norm_rope_kv_write(const void *q, const void *k, const void *v, const void *q_norm_weight,
                                   const void *k_norm_weight, float eps, const void *cos_table,
                                   const void *sin_table, int32_t max_position, const int32_t *positions,
                                   const int64_t *slot_mapping, int32_t num_tokens, int32_t num_q_heads,
                                   void *q_out, const pa_kv_pool *pool, pa_stream_t stream) {
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!q || !k || !v || !q_norm_weight || !k_norm_weight || !cos_table || !sin_table || !positions ||
      !slot_mapping || !q_out)
    return PA_ERR_NULL;
  if (num_q_heads < 1 || num_q_heads > 1024 || max_position < 1 || !(eps >= 0.f) || !isfinite(eps))
    return PA_ERR_SHAPE;
  if ((int64_t)num_tokens * (num_q_heads + 2 * pool->num_kv_heads) > INT32_MAX) return PA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q_out) || !aligned16(q_norm_weight) ||
      !aligned16(k_norm_weight) || !aligned16(cos_table) || !aligned16(sin_table) || !aligned4(positions) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PA_ERR_ALIGN;
  DeviceState *d = nullptr;
  if ((st = device_state(&d)) != PA_OK) return st;
  RopeWriteParams p;
  p.q = q;
  p.k = k;
  p.v = v;
  p.q_weight = q_norm_weight;
  p.k_weight = k_norm_weight;
  p.cos_table = cos_table;
  p.sin_table = sin_table;
  p.positions = positions;
  p.slots = slot_mapping;
  p.q_out = q_out;
  p.k_cache = pool->k_cache;
  p.v_cache = pool->v_cache;
  p.err = d->err;
  p.num_slots = (int64_t)pool->num_blocks * kBlock;
  p.num_tokens = num_tokens;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = pool->num_kv_heads;
  p.max_position = max_position;
  p.eps = eps;
  cudaError_t e = launch_rope_write(p, pool->dtype, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_kv_block_copy(const pa_kv_pool *pools, int32_t num_layers, const int32_t *pairs, int32_t num_pairs,
                           pa_stream_t stream) {
  if (num_layers < 0 || num_pairs < 0) return PA_ERR_SHAPE;
  if (num_layers == 0 || num_pairs == 0) return PA_OK;
  if (!pools || !pairs) return PA_ERR_NULL;
  if (!aligned4(pairs)) return PA_ERR_ALIGN;
  for (int32_t l = 0; l < num_layers; ++l) {
    pa_status st = check_pool(&pools[l]);
    if (st != PA_OK) return st;
    if (pools[l].num_blocks != pools[0].num_blocks || pools[l].num_kv_heads != pools[0].num_kv_heads ||
        pools[l].dtype != pools[0].dtype)
      return PA_ERR_SHAPE;
  }
  DeviceState *d = nullptr;
  pa_status st = device_state(&d);
  if (st != PA_OK) return st;
  BlockCopyParams p{};
  p.pairs = pairs;
  p.err = d->err;
  p.num_blocks = pools[0].num_blocks;
  p.block_vecs = kBlock * pools[0].num_kv_heads * kHeadDim * 2 / 16;
  for (int32_t l0 = 0; l0 < num_layers; l0 += kCopyLayers) {  // up to kCopyLayers layers per launch
    const int n = num_layers - l0 < kCopyLayers ? num_layers - l0 : kCopyLayers;
    for (int i = 0; i < n; ++i) {
      p.k[i] = pools[l0 + i].k_cache;
      p.v[i] = pools[l0 + i].v_cache;
    }
    cudaError_t e = launch_block_copy(p, n, num_pairs, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return PA_OK;
}

pa_status pa_selftest_bounded_wait(uint32_t limit_us, pa_stream_t stream) {
  if (limit_us < 1 || limit_us > 2000000) return PA_ERR_SHAPE;
  DeviceState *d = nullptr;
  pa_status st = device_state(&d);
  if (st != PA_OK) return st;
  cudaError_t e = launch_bounded_wait_selftest(d->err, (uint64_t)limit_us * 1000ull, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

pa_status pa_get_device_error(pa_stream_t stream, int32_t *detail) {
  DeviceState *d = nullptr;
  pa_status st = device_state(&d);
  if (st != PA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int host[2] = {0, 0};
  cudaError_t e = cudaMemcpyAsync(host, d->err, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(d->err, 0, sizeof(host), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e);
  if (detail) *detail = host[1];
  return static_cast<pa_status>(host[0]);
}

// ---- one persistent launch for a mixed step --------------------------------------

namespace {
constexpr size_t kMixedSyncBytes = 256;  // the launch's 4 counters, then the decode's workspace
constexpr int kMixedMaxSeqs = 6000;
constexpr int kMixedMaxChunks = 256;
}  // namespace

size_t pa_mixed_step_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads) {
  if (num_seqs < 0 || num_seqs > kMixedMaxSeqs || num_kv_heads < 1 || num_q_heads < 1 ||
      num_q_heads % num_kv_heads != 0)
    return 0;
  return kMixedSyncBytes + decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads);
}

pa_status pa_mixed_step(const pa_kv_pool *pool, int32_t num_q_heads, float scale, const void *k_chunks,
                        const void *v_chunks, const int64_t *chunk_slots, int32_t num_chunk_tokens,
                        const void *q_chunks, const int32_t *chunk_starts, const int32_t *chunk_lens,
                        const int32_t *chunk_block_tables, int32_t chunk_max_blocks,
                        const int32_t *chunk_context_lens, int32_t num_chunks, int32_t total_q_tokens,
                        int32_t max_chunk_len, void *out_chunks, const void *q, const void *k_dec, const void *v_dec,
                        const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                        int32_t num_seqs, void *out, void *workspace, size_t workspace_bytes, pa_stream_t stream) {
  const int num_tokens = num_chunk_tokens;
  const void *k_new = k_chunks, *v_new = v_chunks;
  const int64_t *slot_mapping = chunk_slots;
  pa_status st = check_pool(pool);
  if (st != PA_OK) return st;
  int group = 0;
  if ((st = check_group(num_q_heads, pool->num_kv_heads, &group)) != PA_OK) return st;
  if (num_tokens < 0 || num_chunks < 0 || num_seqs < 0 || num_chunks > kMixedMaxChunks ||
      num_seqs > kMixedMaxSeqs || num_seqs > mixed_max_seqs(group))
    return PA_ERR_SHAPE;
  if (num_tokens == 0 && num_chunks == 0 && num_seqs == 0) return PA_OK;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_SHAPE;
  if (num_tokens > 0) {
    if (!k_new || !v_new || !slot_mapping) return PA_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u)) return PA_ERR_ALIGN;
  }
  if (num_chunks > 0) {
    if (!q_chunks || !chunk_starts || !chunk_lens || !chunk_block_tables || !chunk_context_lens || !out_chunks)
      return PA_ERR_NULL;
    if (max_chunk_len < 1 || max_chunk_len > PA_MAX_CHUNK_LEN || chunk_max_blocks < 1 || total_q_tokens < 1)
      return PA_ERR_SHAPE;
    if (!aligned16(q_chunks) || !aligned16(out_chunks) || !aligned4(chunk_block_tables) ||
        !aligned4(chunk_context_lens) || !aligned4(chunk_starts) || !aligned4(chunk_lens))
      return PA_ERR_ALIGN;
  }
  if (num_seqs > 0) {
    if (!q || !block_tables || !context_lens || !out || (k_dec == nullptr) != (v_dec == nullptr)) return PA_ERR_NULL;
    if (max_blocks_per_seq < 1) return PA_ERR_SHAPE;
    if (!aligned16(q) || !aligned16(out) || !aligned4(block_tables) || !aligned4(context_lens) ||
        (k_dec && (!aligned16(k_dec) || !aligned16(v_dec))))
      return PA_ERR_ALIGN;
  }
  if (!workspace) return PA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return PA_ERR_ALIGN;
  if (workspace_bytes < pa_mixed_step_workspace_bytes(num_seqs, num_q_heads, pool->num_kv_heads))
    return PA_ERR_WORKSPACE;
  DeviceState *d = nullptr;
  if ((st = device_state(&d)) != PA_OK) return st;

  MixedParams mp{};
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  mp.sync = reinterpret_cast<int32_t *>(ws);
  // the write
  mp.w.k = k_new;
  mp.w.v = v_new;
  mp.w.slots = slot_mapping;
  mp.w.k_cache = pool->k_cache;
  mp.w.v_cache = pool->v_cache;
  mp.w.num_slots = (int64_t)pool->num_blocks * kBlock;
  mp.w.num_tokens = num_tokens;
  mp.w.row_vecs = pool->num_kv_heads * kHeadDim * 2 / 16;
  mp.w.err = d->err;
  // the prefill (no window, the plain per-tile schedule)
  PrefillParams &pp = mp.pp;
  pp.q = q_chunks;
  pp.k_cache = pool->k_cache;
  pp.v_cache = pool->v_cache;
  pp.chunk_starts = chunk_starts;
  pp.chunk_lens = chunk_lens;
  pp.block_tables = chunk_block_tables;
  pp.context_lens = chunk_context_lens;
  pp.out = out_chunks;
  pp.err = d->err;
  pp.max_blocks_per_seq = chunk_max_blocks;
  pp.num_chunks = num_chunks;
  pp.num_kv_heads = pool->num_kv_heads;
  pp.num_q_heads = num_q_heads;
  pp.num_blocks = pool->num_blocks;
  pp.total_q_tokens = total_q_tokens;
  pp.max_chunk_len = num_chunks > 0 ? max_chunk_len : 1;
  pp.scale_log2 = scale * 1.4426950408889634f;
  // the decode (split items merged in the launch)
  DecodeParams &dp = mp.dp;
  if (!decode_workspace_carve(ws + kMixedSyncBytes, workspace_bytes - kMixedSyncBytes, num_seqs, num_q_heads,
                              pool->num_kv_heads, dp))
    return PA_ERR_WORKSPACE;
  dp.meta = nullptr;
  dp.counters = reinterpret_cast<int32_t *>(
      ws + kMixedSyncBytes + decode_workspace_counters_offset(num_seqs, num_q_heads, pool->num_kv_heads));
  dp.q = q;
  dp.block_tables = block_tables;
  dp.context_lens = context_lens;
  dp.out = out;
  dp.err = d->err;
  dp.k_new = num_seqs > 0 ? k_dec : nullptr;  // each sequence's new token, written as its page is read
  dp.v_new = num_seqs > 0 ? v_dec : nullptr;
  dp.k_pool = pool->k_cache;
  dp.v_pool = pool->v_cache;
  dp.max_blocks_per_seq = num_seqs > 0 ? max_blocks_per_seq : 1;
  dp.num_seqs = num_seqs;
  dp.num_kv_heads = pool->num_kv_heads;
  dp.num_q_heads = num_q_heads;
  dp.num_blocks = pool->num_blocks;
  dp.scale_log2 = pp.scale_log2;

  CUtensorMap maps[6];
  memset(maps, 0, sizeof(maps));
  if (!pool_map(&maps[0], pool, pool->k_cache, false) || !pool_map_vpages(&maps[1], pool, pool->v_cache) ||
      !pool_map(&maps[4], pool, pool->k_cache, true) || !pool_map(&maps[5], pool, pool->v_cache, true))
    return PA_ERR_CUDA;
  if (num_chunks > 0 &&
      !query_maps(&maps[2], &maps[3], q_chunks, out_chunks, pool->dtype, num_q_heads, total_q_tokens, group))
    return PA_ERR_CUDA;
  cudaError_t e = launch_mixed(mp, maps, pool->dtype, group, static_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported || e == cudaErrorCooperativeLaunchTooLarge) return PA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // extern "C"

