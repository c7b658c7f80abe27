// Launchers of the paged decode (the kernels themselves: decode_kernel.cuh),
// the one-cluster-per-item kernel and the combine of split items.
#include "decode_kernel.cuh"

namespace pa {
namespace {

// Log-sum-exp merge of the fragments of every item a single warp did not finish.
// One warp per (sequence, query head).
template <typename T, int G>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p) {
  griddep_wait();
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (gw < p.num_seqs * p.num_q_heads) {
    const int s = gw / p.num_q_heads, qh = gw % p.num_q_heads;
    const int h = qh / G, gg = qh % G;
    const int hkv = p.num_kv_heads;
    const int pages = p.meta[s + 1] - p.meta[s];
    const int64_t P = (int64_t)p.meta[p.num_seqs] * hkv;
    const int64_t W = P < p.num_workers ? P : p.num_workers;
    const int64_t A = (int64_t)hkv * p.meta[s] + (int64_t)h * pages;
    const int wf = pages ? worker_of(A, P, W) : 0;
    const int wl = pages ? worker_of(A + pages - 1, P, W) : 0;
    if (pages != 0 && wf != wl)  // otherwise the split kernel wrote this output directly
      merge_fragments<T, G, 32>(p, s, h, gg, wf, wl - wf + 1, lane);
  }
  griddep_launch_dependents();
}

// ---- one cluster per item (few items: every item gets one or two SMs) ------------
// The item's pages are dealt round-robin to the kItemWarps warps of each CTA of
// a cluster of 1 or 2 CTAs, each warp streaming its pages through its own TMA
// ring (two CTAs double the bytes in flight for the item).  Each CTA then
// merges its warps' states (m, l, o) in its own shared memory (reusing the
// stage buffers), all threads at once; CTA 1 stores its merged state into CTA
// 0's shared memory through the cluster and exits, and CTA 0 merges the two
// and writes the item's output.  No workspace and no second kernel.
constexpr int kItemWarps = 8;

template <typename T, int G, bool Q8, bool F8>
__global__ void __launch_bounds__(kItemWarps * 32, 1)
decode_item_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                   const DecodeParams p) {
  using Ly = Layout<G>;
  constexpr int NQ = Ly::NQ, DPL = Ly::DPL;
  constexpr int kMerge = 4 + kHeadDim;  // floats per (warp, head): m, l, 2 unused, o[128] (16-byte aligned)
  // full 8 KB stages for int8 too: a larger footprint keeps one CTA per SM, so
  // the two CTAs of an item (and different items) never share an SM's copy engine
  constexpr int SST = STAGE;
  static_assert(G * kMerge * 4 <= kStages * SST, "merge buffer fits a warp's stages");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *stages = smem + warp * kStages * SST;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kItemWarps * kStages * SST) + warp * kStages;
  float2 *pbuf2 = reinterpret_cast<float2 *>(smem + kItemWarps * kStages * SST + kItemWarps * kStages * 8) +
                  warp * 16 * G;
  // CTA 0 only: CTA 1's merged state, [G][kMerge] floats
  float *peer = reinterpret_cast<float *>(smem + kItemWarps * kStages * SST + kItemWarps * kStages * 8 +
                                          kItemWarps * 16 * G * 8);

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
  }

  const int ncta = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
  const int item = blockIdx.x / ncta;
  const int hkv = p.num_kv_heads;
  const int s = item / hkv, h = item % hkv;
  // Warp gw of the item's nw warps takes the visible pages gw, gw + nw, gw +
  // 2 nw, ... (counted from the first page of the sliding window, if any):
  // without a window its first block ids do not depend on the length, so the
  // length and the block ids are fetched at once.  No kernel of this library writes the block
  // tables or the lengths, so they are read before waiting for the previous
  // kernel (that wait covers the pool, which a KV write fills, and q, which may
  // be another call's output); their latency overlaps the previous kernel.
  const int gw = rank * kItemWarps + warp, nw = ncta * kItemWarps;
  const int32_t *bt = p.block_tables + (int64_t)s * p.max_blocks_per_seq;
  const int ctx = __ldg(p.context_lens + s);
  int win_base = 0;  // window of 32 block ids: lane j holds page gw + nw (win_base + j)
  int32_t win = (gw + nw * lane < p.max_blocks_per_seq) ? __ldg(bt + gw + nw * lane) : -1;
  const bool ctx_ok = ctx >= 1 && ctx <= p.max_blocks_per_seq * kBlock;  // uniform over the cluster
  const int lo = ctx_ok ? window_lo(ctx, p.window) : 0, first = lo / kBlock;  // first visible key, its page
  const int pages = ctx_ok ? (ctx + kBlock - 1) / kBlock - first : 0;         // visible pages
  const int n = pages > gw ? (pages - gw + nw - 1) / nw : 0;                  // pages of this warp
  if (first != 0) win = (gw + nw * lane < pages) ? __ldg(bt + first + gw + nw * lane) : -1;

  uint32_t bad_mask = 0;
  auto issue = [&](int i, int st) {
    if ((i & ~31) != win_base) {
      win_base = i & ~31;
      const int pj = gw + nw * (win_base + lane);
      win = (pj < pages) ? __ldg(bt + first + pj) : -1;
    }
    const int blk = __shfl_sync(FULL, win, i & 31);
    const bool ok = (unsigned)blk < (unsigned)p.num_blocks;
    if (lane == 0) {
      if (ok) {
        load_page<Q8>(stages + st * SST, &kmap, &vmap, &bars[st], p, h, blk);
      } else {
        set_error(p.err, PA_ERR_RANGE, s);
        mbar_arrive(&bars[st]);
      }
    }
    bad_mask = ok ? (bad_mask & ~(1u << st)) : (bad_mask | (1u << st));
  };

  // With early_pages the caller guarantees that the kernels still running
  // (the one before this one and, behind a KV write, the one before that)
  // write no page of the sequence but the last visible one (a decode step's
  // KV write touches only the new token's page), so the first stages of the
  // other pages are fetched before the wait and overlap those kernels.
  const int npre = n < kStages ? n : kStages;
  uint32_t deferred = (1u << npre) - 1u;
  if (p.early_pages) {
    for (int i = 0; i < npre; ++i) {
      if (gw + nw * i != pages - 1) {
        issue(i, i);
        deferred &= ~(1u << i);
      }
    }
  }
  griddep_wait();
  for (int i = 0; i < npre; ++i)
    if ((deferred >> i) & 1u) issue(i, i);

  QReg<Q8 && !F8> q[G][DPL / 2];
  float qsc[G];
  float2 o[G][2];
  float m[G], l[G];
  {
    const T *qp = reinterpret_cast<const T *>(p.q) + ((int64_t)s * p.num_q_heads + (int64_t)h * G) * kHeadDim;
    load_q<T, G, Q8 && !F8>(qp, p.scale_log2, lane, q, qsc);
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      m[gg] = -INFINITY;
      l[gg] = 0.f;
      o[gg][0] = make_float2(0.f, 0.f);
      o[gg][1] = make_float2(0.f, 0.f);
    }
  }
  if (!ctx_ok) {  // nothing was issued (n = 0); output untouched
    if (h == 0 && rank == 0 && threadIdx.x == 0) set_error(p.err, PA_ERR_RANGE, s);
    griddep_launch_dependents();
    return;
  }

  bool timed_out = false;
  for (int i = 0; i < n; ++i) {
    const int st = i % kStages;
    if (!mbar_wait(&bars[st], (uint32_t)((i / kStages) & 1))) {
      if (lane == 0) set_error(p.err, PA_ERR_TIMEOUT, s);
      // give the copies still in flight a short, bounded chance to land
      for (int r = i + 1; r < (n < i + kStages ? n : i + kStages); ++r)
        mbar_wait(&bars[r % kStages], (uint32_t)((r / kStages) & 1), kWaitLimitNs / 8);
      timed_out = true;
      break;
    }
    if (!((bad_mask >> st) & 1u)) {
      const int pg = gw + nw * i;                              // visible page
      const int nv = min(kBlock, ctx - (first + pg) * kBlock);  // keys of the sequence in this page
      if constexpr (!Q8) {
        if (p.k_new && pg == pages - 1) {  // the page of the sequence's new token (the warp's last page)
          append_row<T>(stages + st * SST, p, s, h, __ldg(bt + first + pg), nv - 1, lane);
          fence_proxy_async_smem();
        }
      }
      decode_page<T, G, Q8, F8>(stages + st * SST, pg == 0 ? lo - first * kBlock : 0, nv, q, qsc, o, m, l, pbuf2,
                            lane);
    }
    __syncwarp();  // every lane is done with this stage and with pbuf
    if (i + kStages < n) issue(i + kStages, st);
  }

  // the next kernel may start its set-up while the item is merged (it still
  // waits for this grid to complete before reading anything)
  griddep_launch_dependents();
  // ---- merge: the warps of each CTA in its shared memory (the stage buffers
  // are idle now), then CTA 1's state into CTA 0 through the cluster ----
  __syncthreads();
  float *mine = reinterpret_cast<float *>(stages);
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    float lt = l[gg];
#pragma unroll
    for (int off = NQ; off < 32; off <<= 1) lt += __shfl_xor_sync(FULL, lt, off);
    float *dst = mine + gg * kMerge;
    if (lane == 0) {
      dst[0] = m[gg];
      dst[1] = lt;
    }
    *reinterpret_cast<float4 *>(dst + 4 + 4 * lane) = make_float4(o[gg][0].x, o[gg][0].y, o[gg][1].x, o[gg][1].y);
  }
  const bool any_timeout = __syncthreads_or(timed_out ? 1 : 0) != 0;
  // thread (warp mg, lane) merges head mg, dims 4 lane .. 4 lane + 3, over the CTA's warps in order
  const int mg = warp;
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  if (mg < G) {
    float mv[kItemWarps], lv[kItemWarps];
    float4 ov[kItemWarps];
#pragma unroll
    for (int w = 0; w < kItemWarps; ++w) {  // every load first (they are independent), then the arithmetic
      const float *a = reinterpret_cast<const float *>(smem + w * kStages * SST) + mg * kMerge;
      mv[w] = a[0];
      lv[w] = a[1];
      ov[w] = *reinterpret_cast<const float4 *>(a + 4 + 4 * lane);
    }
#pragma unroll
    for (int w = 0; w < kItemWarps; ++w) M = fmaxf(M, mv[w]);
#pragma unroll
    for (int w = 0; w < kItemWarps; ++w) {
      const float wgt = (mv[w] == -INFINITY) ? 0.f : exp2f(mv[w] - M);  // a warp without pages: weight 0
      L += lv[w] * wgt;
      O.x = fmaf(wgt, ov[w].x, O.x);
      O.y = fmaf(wgt, ov[w].y, O.y);
      O.z = fmaf(wgt, ov[w].z, O.z);
      O.w = fmaf(wgt, ov[w].w, O.w);
    }
  }
  if (ncta > 1) {
    if (rank != 0) {  // hand the state to CTA 0 and leave
      if (mg < G) {
        const uint32_t dst = map_to_rank(peer + mg * kMerge, 0);
        if (lane == 0) {
          st_cluster_f32(dst, M);
          st_cluster_f32(dst + 4, L);
        }
        st_cluster_v4(dst + 4 * (4 + 4 * lane), O);
      }
      cluster_arrive();  // release: CTA 0 sees the stores once its wait returns
      return;
    }
    cluster_arrive();
    cluster_wait();
    if (mg < G) {
      const float *a = peer + mg * kMerge;
      const float M1 = a[0], L1 = a[1];
      const float4 O1 = *reinterpret_cast<const float4 *>(a + 4 + 4 * lane);
      const float Mx = fmaxf(M, M1);
      const float w0 = (M == -INFINITY) ? 0.f : exp2f(M - Mx), w1 = (M1 == -INFINITY) ? 0.f : exp2f(M1 - Mx);
      L = L * w0 + L1 * w1;
      O = make_float4(fmaf(w1, O1.x, O.x * w0), fmaf(w1, O1.y, O.y * w0), fmaf(w1, O1.z, O.z * w0),
                      fmaf(w1, O1.w, O.w * w0));
    }
  }
  if (mg < G && !any_timeout) {
    const float inv = 1.f / L;
    T *op = reinterpret_cast<T *>(p.out) + ((int64_t)s * p.num_q_heads + h * G + mg) * kHeadDim + 4 * lane;
    uint2 pk;
    pk.x = Pack<T>::from_f2(O.x * inv, O.y * inv);
    pk.y = Pack<T>::from_f2(O.z * inv, O.w * inv);
    *reinterpret_cast<uint2 *>(op) = pk;
  }
}

int item_smem_bytes(int group) {
  return 1024 + kItemWarps * kStages * STAGE + kItemWarps * kStages * 8 + kItemWarps * 16 * group * 8 +
         group * (4 + kHeadDim) * 4;
}

int split_smem_bytes(int group, int num_seqs, bool q8) {
  const int sst = q8 ? stage_stride<true>() : stage_stride<false>();
  return 1024 + NW * kStages * sst + NW * kStages * 8 + NW * 16 * group * 8 + (num_seqs + 1) * 4;
}

}  // namespace

// A cluster per item pays off when every item gets its own SMs (two when they
// fit) and the longest item the length bound allows, streamed by them, still
// ends before the split path would end in its best case, that item alone
// spread over all SMs (the batch may be that skewed: only the bound is known
// on the host).  The split path pays a second launch and a merge through
// global memory.  Rates are round measured figures for this part: ~150 GB/s
// per SM for TMA page streams, ~6 TB/s of HBM for the whole GPU.  Returns the
// CTAs per item (1 or 2), or 0 for the split path.
int decode_item_ctas(int items, int max_pages_per_item) {
  const int sms = sm_count();
  if (items > sms) return 0;
  const int ctas = 2 * items <= sms ? 2 : 1;
  const double item_bytes = (double)max_pages_per_item * 2.0 * kBlock * kHeadDim * 2;
  const double item_us = 3.0 + item_bytes / (ctas * 150e3);
  const double split_us = 8.0 + item_bytes / 6e6;
  return item_us < split_us ? ctas : 0;
}

namespace {

template <typename T, int G, bool Q8, bool F8>
cudaError_t launch_typed(const DecodeParams &p0, const CUtensorMap &kmap, const CUtensorMap &vmap,
                         int max_workers, int max_pages_per_item, cudaStream_t stream) {
  DecodeParams p = p0;
  const int items = p.num_seqs * p.num_kv_heads;
  const int ctas = p.counters ? 0 : decode_item_ctas(items, max_pages_per_item);
  if (ctas > 0) {
    const int ismem = item_smem_bytes(G);
    static KernelSetup item_setup;
    cudaError_t e = kernel_setup(item_setup, decode_item_kernel<T, G, Q8, F8>, ismem, kItemWarps * 32, nullptr);
    if (e != cudaSuccess) return e;
    return launch_pdl_cluster(decode_item_kernel<T, G, Q8, F8>, dim3(items * ctas), dim3(kItemWarps * 32), ismem, ctas,
                              stream, kmap, vmap, p);
  }
  const int smem = split_smem_bytes(G, p.num_seqs, Q8);
  // Per instantiation: raise the dynamic shared-memory limit and cache the
  // occupancy for the largest size seen (launch-time API calls stay out of
  // the hot path and out of CUDA-graph capture after the first call).
  static KernelSetup split_setup;
  int per_sm = 0;
  cudaError_t e = kernel_setup(split_setup, decode_split_kernel<T, G, Q8, F8>, smem, NW * 32, &per_sm);
  if (e != cudaSuccess) return e;
  int grid = sm_count() * per_sm;
  const int want = (max_workers + NW - 1) / NW;
  if (want < grid) grid = want;
  if (grid < 1) grid = 1;
  if (grid * NW > kDecodeMaxWorkers) grid = kDecodeMaxWorkers / NW;
  p.num_workers = grid * NW;
  e = launch_pdl(decode_split_kernel<T, G, Q8, F8>, dim3(grid), dim3(NW * 32), smem, stream, kmap, vmap, p);
  if (e != cudaSuccess) return e;
  if (p.counters) return cudaSuccess;  // the split kernel merged the split items itself
  const int cgrid = (p.num_seqs * p.num_q_heads + 3) / 4;
  return launch_pdl(decode_combine_kernel<T, G>, dim3(cgrid), dim3(128), 0, stream, p);
}

}  // namespace

size_t decode_workspace_counters_offset(int num_seqs, int num_q_heads, int num_kv_heads) {
  const int group = num_q_heads / num_kv_heads;
  const size_t slots = (size_t)num_seqs * num_kv_heads + kDecodeMaxWorkers;
  const size_t meta = (((size_t)num_seqs + 1) * 4 + 255) & ~(size_t)255;
  const size_t ml = (slots * group * 2 * 4 + 255) & ~(size_t)255;
  const size_t o = slots * group * kHeadDim * 4;
  return meta + ml + o;
}

// page prefix, (m, l) and o partials, then one counter per (sequence, KV head) item
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads) {
  const size_t counters = ((size_t)num_seqs * num_kv_heads * 4 + 255) & ~(size_t)255;
  return decode_workspace_counters_offset(num_seqs, num_q_heads, num_kv_heads) + counters;
}

bool decode_workspace_carve(void *ws, size_t bytes, int num_seqs, int num_q_heads, int num_kv_heads,
                            DecodeParams &p) {
  if (bytes < decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads)) return false;
  const int group = num_q_heads / num_kv_heads;
  const size_t slots = (size_t)num_seqs * num_kv_heads + kDecodeMaxWorkers;
  uint8_t *b = static_cast<uint8_t *>(ws);
  const size_t meta = (((size_t)num_seqs + 1) * 4 + 255) & ~(size_t)255;
  const size_t ml = (slots * group * 2 * 4 + 255) & ~(size_t)255;
  p.meta = reinterpret_cast<int32_t *>(b);
  p.ws_ml = reinterpret_cast<float *>(b + meta);
  p.ws_o = reinterpret_cast<float *>(b + meta + ml);
  return true;
}

cudaError_t launch_decode(const DecodeParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                          int dtype, int group, int max_workers, int max_pages_per_item, bool q8, bool f8,
                          cudaStream_t stream) {
#define PA_DECODE_CASE(T, G)                                                                    \
  if (group == G)                                                                               \
    return f8   ? launch_typed<T, G, true, true>(p, kmap, vmap, max_workers, max_pages_per_item, stream)  \
           : q8 ? launch_typed<T, G, true, false>(p, kmap, vmap, max_workers, max_pages_per_item, stream) \
                : launch_typed<T, G, false, false>(p, kmap, vmap, max_workers, max_pages_per_item, stream);
  if (dtype == PA_BF16) {
    PA_DECODE_CASE(__nv_bfloat16, 1)
    PA_DECODE_CASE(__nv_bfloat16, 2)
    PA_DECODE_CASE(__nv_bfloat16, 4)
    PA_DECODE_CASE(__nv_bfloat16, 8)
  } else {
    PA_DECODE_CASE(__half, 1)
    PA_DECODE_CASE(__half, 2)
    PA_DECODE_CASE(__half, 4)
    PA_DECODE_CASE(__half, 8)
  }
#undef PA_DECODE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
