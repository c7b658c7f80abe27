// Internal interface between the C-ABI layer (pa_abi.cu) and the kernel
// translation units.  Not installed; not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "../../include/pagedattn.h"

namespace pa {

// Every bounded wait gives up after this long (then PA_ERR_TIMEOUT).
constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;

constexpr int kHeadDim = 128;
constexpr int kBlock = 16;

// ---- kv_cache_write ------------------------------------------------------------
struct WriteParams {
  const void *k;
  const void *v;
  const int64_t *slots;
  void *k_cache;
  void *v_cache;
  int64_t num_slots;   // num_blocks * 16
  int32_t num_tokens;
  int32_t row_vecs;    // 16-byte vectors per token row = Hkv * 128 * 2 / 16
  int *err;
};
cudaError_t launch_kv_write(const WriteParams &p, cudaStream_t stream);

// Quantising write into an int8 pool: one fp32 scale per (token, KV head) for
// K and for V, codes int8 [num_blocks][16][Hkv][128], scales [num_blocks][Hkv][16].
struct WriteQ8Params {
  const void *k;             // [T][Hkv][128] in `dtype`
  const void *v;
  const int64_t *slots;
  int8_t *k_cache;
  int8_t *v_cache;
  float *k_scale;
  float *v_scale;
  int64_t num_slots;
  int32_t num_tokens;
  int32_t num_kv_heads;
  int *err;
};
// f8: E4M3 codes with scale = max |x| / 448 + 1e-8 instead of int8 codes.
cudaError_t launch_kv_write_q8(const WriteQ8Params &p, int dtype, bool f8, cudaStream_t stream);

// ---- q/k RMSNorm + rotary embedding fused into the KV write -------------------------------
struct RopeWriteParams {
  const void *q;             // [T][Hq][128]
  const void *k;             // [T][Hkv][128]
  const void *v;
  const void *q_weight;      // [128]
  const void *k_weight;
  const void *cos_table;     // [max_position][128]
  const void *sin_table;
  const int32_t *positions;  // [T]
  const int64_t *slots;      // [T]
  void *q_out;               // [T][Hq][128]
  void *k_cache;
  void *v_cache;
  int *err;
  int64_t num_slots;
  int32_t num_tokens;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t max_position;
  float eps;
};
cudaError_t launch_rope_write(const RopeWriteParams &p, int dtype, cudaStream_t stream);

// ---- self-test of the bounded waits --------------------------------------------------------
cudaError_t launch_bounded_wait_selftest(int *err, uint64_t limit_ns, cudaStream_t stream);

// ---- copy-on-write block copy ---------------------------------------------------------
constexpr int kCopyLayers = 64;          // layer pools per launch
struct BlockCopyParams {
  void *k[kCopyLayers];                  // per layer: pool base addresses
  void *v[kCopyLayers];
  const int32_t *pairs;                  // [num_pairs][2] (src, dst)
  int *err;
  int32_t num_blocks;
  int32_t block_vecs;                    // 16-byte vectors per block (16 * Hkv * 128 * 2 / 16)
};
cudaError_t launch_block_copy(const BlockCopyParams &p, int num_layers, int num_pairs, cudaStream_t stream);

// ---- decode (split-K over a balanced page range per warp) -----------------------
constexpr int kDecodeWarps = 4;         // warps per CTA; each warp is an independent worker
constexpr int kDecodeMaxWorkers = 8192; // upper bound on workers (warps) per launch
constexpr int kDecodeStageBytes = 8192; // one 16-token page of K and V for one KV head

struct DecodeParams {
  const void *q;             // [S][Hq][128]
  const int32_t *block_tables;
  const int32_t *context_lens;
  void *out;                 // [S][Hq][128]
  int32_t *meta;             // workspace: page prefix over sequences [S + 1]
  float *ws_ml;              // workspace: (m, l) per partial slot and head of the group
  float *ws_o;               // workspace: o[128] per partial slot and head of the group
  int *err;
  const float *k_scale;      // int8 pools only: [num_blocks][Hkv][16] scales of K and V
  const float *v_scale;
  const void *k_new;         // append (16-bit pools only; null: none): each sequence's new token
  const void *v_new;         //   [S][Hkv][128], written at position context_lens[s] - 1
  void *k_pool;              //   pool base addresses for that write
  void *v_pool;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t num_kv_heads;
  int32_t num_q_heads;
  int32_t num_blocks;
  int32_t num_workers;       // warps in the launch
  int32_t window;            // sliding window in keys (0: none)
  int32_t early_pages;       // 1: pages before each sequence's last one are not written by the previous
                             //    kernel, so the one-launch decode fetches them before its dependency wait
  int32_t *counters;         // workspace: arrivals per (sequence, KV head) item; non-null only when the
                             //    caller keeps them zero between calls: the split kernel then merges each
                             //    split item itself (the last fragment to arrive), with no combine launch
  float scale_log2;          // scale * log2(e)
};

struct DecodeLaunch {
  int grid;          // CTAs
  int smem_bytes;    // dynamic shared memory per CTA
};

// Plans and launches the decode: one CTA per (sequence, KV head) item when the
// items are few, else the split and combine kernels.  `group` = Hq / Hkv;
// max_pages_per_item bounds each item's pages (from the host-side max length);
// q8: the pool holds 8-bit codes with per-token scales (p.k_scale, p.v_scale):
// int8 integers, or E4M3 numbers when f8.
// With p.counters set, the split kernel runs alone (whatever the item count)
// and merges split items itself.
cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                          int dtype, int group, int max_workers, int max_pages_per_item, bool q8, bool f8,
                          cudaStream_t stream);
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads);
// Offset and size of the item counters inside the workspace.
size_t decode_workspace_counters_offset(int num_seqs, int num_q_heads, int num_kv_heads);
// CTAs per item of the one-launch decode (1 or 2), or 0 when the split path runs.
int decode_item_ctas(int items, int max_pages_per_item);
// Carves the workspace into meta / ml / o; returns false if it is too small.
bool decode_workspace_carve(void *ws, size_t bytes, int num_seqs, int num_q_heads, int num_kv_heads,
                            DecodeParams &p);

// ---- chunked prefill (tcgen05 tensor cores) -------------------------------------
struct PrefillParams {
  const void *q;             // [rows][Hq][128]
  const void *k_cache;       // pool [num_blocks][16][Hkv][128]
  const void *v_cache;
  const int32_t *chunk_starts;
  const int32_t *chunk_lens;
  const int32_t *block_tables;
  const int32_t *context_lens;
  void *out;
  int *err;
  int32_t max_blocks_per_seq;
  int32_t num_chunks;
  int32_t num_kv_heads;
  int32_t num_q_heads;
  int32_t num_blocks;
  int32_t total_q_tokens;
  int32_t max_chunk_len;
  int32_t window;            // sliding window in keys (0: none)
  float scale_log2;
  // 8-bit pools only: the codes' fp32 scales [num_blocks][Hkv][16]
  const float *k_scale;
  const float *v_scale;
  // balanced (persistent) launch only: a workspace the caller keeps zero-filled
  // between calls (prefill_workspace_bytes); all null for the plain launch
  int32_t *ws_counters;      // arrivals per query tile [num_chunks][Hkv][max_tiles]
  float2 *ws_ml;             // per partial slot and row: (max, sum) of a piece of a split query tile
  float *ws_o;               // per partial slot, row and dim: that piece's unnormalised output
  int32_t max_tiles;         // query tiles per chunk and KV head at most: ceil(max_chunk_len / (128 / G))
};
// Workspace of the balanced prefill for `sms` CTAs.
size_t prefill_workspace_bytes(int num_chunks, int num_q_heads, int num_kv_heads, int max_chunk_len, int sms);
// Carves the workspace into p.ws_* (and sets p.max_tiles); false if it is too small.
bool prefill_workspace_carve(void *ws, size_t bytes, int num_chunks, int num_q_heads, int num_kv_heads,
                             int max_chunk_len, int sms, PrefillParams &p);
// The balanced launch takes at most this many chunks per call.
constexpr int kMaxChunksBalanced = 256;
// omap: `out` as the 3-D tensor {dim, query head, token} with qmap's boxes (for
// the TMA store of whole query tiles).  With p.ws_counters set the balanced
// (persistent) kernel runs: one CTA per SM, key tiles dealt evenly.
cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const CUtensorMap &qmap, const CUtensorMap &omap, int dtype, int group,
                           cudaStream_t stream);

// Chunked prefill over an 8-bit pool (int8 codes, or E4M3 with f8) on the
// tcgen05 tensor cores: kmap / vmap as for the 8-bit decode (one 2 KB box per
// page of one KV head), the scales in p.k_scale / p.v_scale, qmap / omap as
// for launch_prefill; q and out of type `dtype`; no window, no workspace.
cudaError_t launch_prefill8(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                            const CUtensorMap &qmap, const CUtensorMap &omap, int dtype, int group, bool f8,
                            cudaStream_t stream);

// ---- one persistent launch for a mixed step (16-bit pools) ---------------------
// The step's KV write (w), its chunks' prefill (pp: no window, no workspace)
// and its sequences' decode (dp: counters set, split items merged in the
// launch), in one cooperative launch of one CTA per SM.  sync: 4 counters of
// the workspace, zero between calls (each call leaves them zero).
struct MixedParams {
  WriteParams w;
  PrefillParams pp;
  DecodeParams dp;
  int32_t *sync;
};
// maps: prefill K (2 KB half boxes), prefill V (4 KB pages), q, out, decode K,
// decode V (4 KB page boxes).
cudaError_t launch_mixed(const MixedParams &mp, const CUtensorMap *maps, int dtype, int group, cudaStream_t stream);
// Dynamic shared memory of the launch, and the most sequences it takes.
int mixed_smem_bytes(int group, int num_seqs);
int mixed_max_seqs(int group);

// ---- launch helper ------------------------------------------------------------
// Launch with programmatic stream serialization (see griddep_wait()).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Same, with thread-block clusters of `cluster_x` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster_x,
                               cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster_x;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---- shared host helpers (pa_abi.cu) ------------------------------------------
int sm_count();
// pa_paged_attn_decode's argument checks up to (not including) the workspace.
pa_status decode_check_args(const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t max_context_len, float scale, void *out);
// Unique id of the current CUDA context (initialising the current device's
// primary context if none is current).
pa_status current_context_id(unsigned long long *id);
// The context id recorded by the entry point now running on this thread
// (every entry point that launches looks it up first).
unsigned long long launch_context_id();

// A kernel's launch set-up (its raised dynamic shared-memory limit and the
// occupancy at that size) belongs to one context: it is redone when the
// calling thread's context is another one, or a larger size is wanted.
struct KernelSetup {
  std::mutex mutex;
  unsigned long long ctx = 0;
  int smem = 0;
  int per_sm = 0;
};
template <typename Kernel>
cudaError_t kernel_setup(KernelSetup &s, Kernel kernel, int smem, int threads, int *per_sm) {
  std::lock_guard<std::mutex> lock(s.mutex);
  const unsigned long long ctx = launch_context_id();
  if (s.ctx != ctx || smem > s.smem) {
    const int want = (s.ctx == ctx && s.smem > smem) ? s.smem : smem;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, want);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;
    s.ctx = ctx;
    s.smem = want;
    s.per_sm = n;
  }
  if (per_sm) *per_sm = s.per_sm;
  return cudaSuccess;
}
bool encode_tensor_map(CUtensorMap *map, CUtensorMapDataType dtype, int rank, void *base,
                       const uint64_t *dims, const uint64_t *strides_bytes, const uint32_t *box,
                       CUtensorMapSwizzle swizzle,
                       CUtensorMapL2promotion promotion = CU_TENSOR_MAP_L2_PROMOTION_L2_256B);

}  // namespace pa
