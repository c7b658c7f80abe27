// One persistent launch for a mixed chunked-prefill + decode step over a
// 16-bit pool (page "Модуль 04: KV-кэш и арифметика памяти", section 3.4:
// prefill chunks interleaved with the decode of running sequences in one
// step; page "Модуль 12: Финальный проект: мини-движок инференса", "Куда
// расти": production engines fuse the step's attention into dedicated
// kernels).  One CTA of 512 threads per SM, launched cooperatively (every CTA
// resident at once), does the whole step, its CTAs split between two roles by
// a cost model that every CTA evaluates alike from the chunk metadata and the
// context lengths:
//
//   prefill (the first np CTAs): the KV write of the chunks' new tokens (the
//     bit copy of pa_kv_cache_write, spread over the np CTAs); a barrier of
//     the np CTAs (an arrival counter in the workspace, a bounded wait, the
//     last CTA to leave sets it back to zero); then the chunks' query tiles,
//     taken from a shared counter, heaviest chunk and query tile first, each
//     the tcgen05 prefill tile of prefill_kernel.cuh;
//   decode (the other CTAs, at once): the split workers of decode_kernel.cuh
//     (8 warps each, the page ranges spread over all of them), each writing a
//     sequence's new token into the page that holds it as it reads that page
//     (pa_paged_attn_decode_append), the split items merged by their last
//     fragment.
//
// The decode never waits for the chunks' write.  np balances the two: a
// prefill (query tile, key tile) pair costs about as much SM time as 3.5
// page-heads of decode (0.75 µs against 0.22 µs per SM for each kernel alone)
// and a query tile's set-up, first loads and epilogue, which a prefill CTA
// running tiles one after another does not hide, about 64 (swept on the
// mixed step); np / grid is the prefill's share of the weighted work.  The
// decode is HBM-bound and the prefill tensor-bound, so side by side the two
// overlap.
#include "decode_kernel.cuh"
#include "prefill_kernel.cuh"

namespace pa {
namespace {

constexpr int kMixedDecodeWarps = 8;       // split workers per decode CTA (the other warps idle)
constexpr float kPairCost = 3.5f;          // one prefill (query tile, key tile) pair, in decode page-heads
constexpr float kTileCost = 64.f;          // one prefill query tile's set-up, first loads and epilogue, likewise
constexpr int kRegsDecode = 232, kRegsIdle = 24;
// the prefill tiles' split here: the loaders keep the tile loop's state too
constexpr int kRegsPrefillSoftmax = 184, kRegsPrefillOther = 72;
static_assert(2 * 128 * kRegsDecode + 2 * 128 * kRegsIdle <= 65536, "register split fits the launch");

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Key tiles of one query tile without a window (from key tile 0 to the tile
// holding its last row's last key).
__device__ __forceinline__ int pairs_of_tile(int start, int ctx, int t0, int TQ) {
  return min(start + t0 + TQ - 1, ctx - 1) / 128 + 1;
}

template <typename T, int G>
__global__ void __launch_bounds__(kThreads, 1)
mixed_step_kernel(const __grid_constant__ CUtensorMap kmap_p, const __grid_constant__ CUtensorMap vmap_p,
                  const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
                  const __grid_constant__ CUtensorMap kmap_d, const __grid_constant__ CUtensorMap vmap_d,
                  const MixedParams mp) {
  constexpr int TQ = 128 / G;
  using Sm = SplitSmem<false, G, kMixedDecodeWarps>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ int warp_tot[kThreads / 32];
  __shared__ int s_tile, s_fail;
  __shared__ unsigned long long s_pairs, s_tiles;
  const int warp = threadIdx.x >> 5;
  const PrefillParams &pp = mp.pp;
  const DecodeParams &dp = mp.dp;
  const int grid = (int)gridDim.x;

  if (threadIdx.x == 0) {
    s_tile = 0;
    s_pairs = 0;
    s_tiles = 0;
  }
  // ---- 1. the split between the roles (the same in every CTA) ----
  int32_t *prefix = reinterpret_cast<int32_t *>(smem + Sm::kPrefixOff);
  scan_pages_n<kThreads>(dp, prefix, warp_tot, (int)blockIdx.x == grid - 1);  // (its barriers order the above)
  const int64_t P = (int64_t)prefix[dp.num_seqs] * dp.num_kv_heads;  // decode page-heads
  const int ntiles = (pp.max_chunk_len + TQ - 1) / TQ;                  // query tiles per chunk bound
  if (threadIdx.x < pp.num_chunks) {  // one thread per chunk (at most 256 chunks)
    const int c = threadIdx.x;
    int row0 = 0;
    unsigned long long pairs = 0, tiles = 0;
    if (tile_rows<G>(pp, c, 0, row0) > 0) {
      const int start = __ldg(pp.chunk_starts + c), len = __ldg(pp.chunk_lens + c);
      for (int t0 = 0; t0 < len; t0 += TQ, ++tiles) pairs += pairs_of_tile(start, start + len, t0, TQ);
    }
    if (pairs) {
      atomicAdd(&s_pairs, pairs * (unsigned long long)pp.num_kv_heads);
      atomicAdd(&s_tiles, tiles * (unsigned long long)pp.num_kv_heads);
    }
  }
  __syncthreads();
  const double wp = (double)kPairCost * (double)s_pairs + (double)kTileCost * (double)s_tiles, wd = (double)P;
  int np = (wp + wd > 0.0) ? (int)(grid * wp / (wp + wd) + 0.5) : 0;
  // at least one prefill CTA when there are chunks (it also reports bad chunk
  // metadata) or chunk tokens to write; at least one decode CTA for pages
  if ((pp.num_chunks > 0 || mp.w.num_tokens > 0) && np < 1) np = 1;
  if (wd > 0.0 && np > grid - 1) np = grid - 1;

  if ((int)blockIdx.x < np) {
    // ---- 2. prefill role: the chunks' new rows (every 16-byte vector, over the np CTAs) ----
    const WriteParams &w = mp.w;
    const int64_t total_v = (int64_t)w.num_tokens * w.row_vecs;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_v; i += (int64_t)np * blockDim.x) {
      const int t = (int)(i / w.row_vecs);
      const int vi = (int)(i - (int64_t)t * w.row_vecs);
      const int64_t slot = __ldg(w.slots + t);
      if (slot < 0 || slot >= w.num_slots) {
        if (vi == 0) set_error(w.err, PA_ERR_RANGE, t);
        continue;
      }
      const uint4 kv = ld_nc_v4(static_cast<const uint4 *>(w.k) + i);
      const uint4 vv = ld_nc_v4(static_cast<const uint4 *>(w.v) + i);
      st_v4(static_cast<uint4 *>(w.k_cache) + slot * w.row_vecs + vi, kv);
      st_v4(static_cast<uint4 *>(w.v_cache) + slot * w.row_vecs + vi, vv);
    }
    // barrier of the np prefill CTAs: every chunk row is written (and visible
    // to the tensor copies) before any query tile reads it
    fence_proxy_async_global();
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
      int fail = 0;
      atomicAdd(mp.sync + 0, 1);
      const uint64_t t_start = globaltimer_ns();
      while (ld_acquire(mp.sync + 0) < np) {
        if (globaltimer_ns() - t_start > kWaitLimitNs) {
          fail = 1;
          break;
        }
        __nanosleep(64);
      }
      // every prefill CTA has arrived once the count reaches np; the last one
      // to leave sets both counts back to zero for the next call
      if (atomicAdd(mp.sync + 1, 1) == np - 1) {
        mp.sync[0] = 0;
        mp.sync[1] = 0;
      }
      if (fail) set_error(w.err, PA_ERR_TIMEOUT, (int)blockIdx.x);
      s_fail = fail;
    }
    __syncthreads();
    if (s_fail) return;  // (reported) the rows may not all be written: no query tile
    fence_proxy_async_global();
    // ---- 3. query tiles from the shared counter until none is left ----
    Bars &bars = *reinterpret_cast<Bars *>(smem + OFF_BAR);
    if (warp == kWarpMma) {
      tc::tmem_alloc(&bars.tmem_base, kTmemCols);
      tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars.tmem_base;
    const int total = pp.num_chunks * pp.num_kv_heads * ntiles;
    for (;;) {
      if (threadIdx.x == 0) s_tile = atomicAdd(mp.sync + 2, 1);
      __syncthreads();
      const int idx = s_tile;
      __syncthreads();  // (s_tile is written again next time round)
      if (idx >= total) break;
      // last chunk first, its last query tile first, KV heads inner
      const int per_chunk = ntiles * pp.num_kv_heads;
      const int c = pp.num_chunks - 1 - idx / per_chunk;
      const int r = idx % per_chunk;
      const int mt = ntiles - 1 - r / pp.num_kv_heads, h = r % pp.num_kv_heads;
      int row0 = 0;
      const int rows = tile_rows<G>(pp, c, mt, row0);
      if (rows < 0 && mt == 0 && h == 0 && threadIdx.x == 0) set_error(pp.err, PA_ERR_RANGE, c);
      if (rows <= 0) continue;
      if (!prefill_tile<T, G, 0, kRegsPrefillSoftmax, kRegsPrefillOther>(kmap_p, vmap_p, qmap, omap, pp, smem, tmem, c,
                                                                          h, mt, row0, true))
        break;
    }
    if (warp == kWarpMma) tc::tmem_dealloc(tmem, kTmemCols);
  } else {
    // ---- decode role: split workers over all decode CTAs (each sequence's new
    // token written into the page that holds it by the worker of that page) ----
    const int64_t W0 = (int64_t)(grid - np) * kMixedDecodeWarps;
    const int64_t W = P < W0 ? P : W0;
    const int64_t w = (int64_t)((int)blockIdx.x - np) * kMixedDecodeWarps + warp;
    if (warp < kMixedDecodeWarps) {
      regs_inc<kRegsDecode>();
      regs_taken();
      if (w < W) decode_split_worker<T, G, false, false, kMixedDecodeWarps>(kmap_d, vmap_d, dp, smem, prefix, warp, w, P, W);
      regs_dec<128>();
    } else {
      regs_dec<kRegsIdle>();
      regs_wait_taken();  // (until then the decode warps' increase may still be waiting for these registers)
      regs_inc<128>();
    }
  }
  // ---- the last CTA to finish sets the tile counter back to zero ----
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(mp.sync + 3, 1) == grid - 1) {
      mp.sync[2] = 0;
      mp.sync[3] = 0;
    }
  }
}

}  // namespace

int mixed_smem_bytes(int group, int num_seqs) {
  const int sst = stage_stride<false>();
  const int decode = 1024 + kMixedDecodeWarps * kStages * sst + kMixedDecodeWarps * kStages * 8 +
                     kMixedDecodeWarps * 16 * group * 8 + (num_seqs + 1) * 4;
  return decode > SMEM_BYTES ? decode : SMEM_BYTES;
}

int mixed_max_seqs(int group) {
  const int sst = stage_stride<false>();
  const int fixed = 1024 + kMixedDecodeWarps * kStages * sst + kMixedDecodeWarps * kStages * 8 +
                    kMixedDecodeWarps * 16 * group * 8;
  return (SMEM_BYTES - fixed) / 4 - 1;
}

namespace {
template <typename T, int G>
cudaError_t launch_mixed_typed(const MixedParams &mp, const CUtensorMap *maps, cudaStream_t stream) {
  static KernelSetup setup;
  const int smem = mixed_smem_bytes(G, mp.dp.num_seqs);
  int per_sm = 0;
  cudaError_t e = kernel_setup(setup, mixed_step_kernel<T, G>, smem, kThreads, &per_sm);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident at once: the grid barrier can complete
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mixed_step_kernel<T, G>, maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], mp);
}
}  // namespace

cudaError_t launch_mixed(const MixedParams &mp, const CUtensorMap *maps, int dtype, int group, cudaStream_t stream) {
#define PA_MIXED_CASE(T, G) \
  if (group == G) return launch_mixed_typed<T, G>(mp, maps, stream);
  if (dtype == PA_BF16) {
    PA_MIXED_CASE(__nv_bfloat16, 1)
    PA_MIXED_CASE(__nv_bfloat16, 2)
    PA_MIXED_CASE(__nv_bfloat16, 4)
    PA_MIXED_CASE(__nv_bfloat16, 8)
  } else {
    PA_MIXED_CASE(__half, 1)
    PA_MIXED_CASE(__half, 2)
    PA_MIXED_CASE(__half, 4)
    PA_MIXED_CASE(__half, 8)
  }
#undef PA_MIXED_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
