// Chunked prefill launchers and the balanced (persistent) variant of the
// per-tile kernel of prefill_kernel.cuh.
#include "prefill_kernel.cuh"

namespace pa {
namespace {


// ============================================================================
// Balanced (persistent) prefill.  One CTA per SM.  The work is the list of
// (query tile, key tile) pairs, numbered chunk by chunk, KV head by KV head,
// query tile by query tile, key tile by key tile; CTA b takes the pairs
// [b W / n, (b + 1) W / n) of the W in all (n CTAs), so every CTA streams the
// same number of key tiles whatever the mix of prefix and chunk lengths (the
// causal mask makes a chunk's last query tiles several times heavier than its
// first ones).  A CTA's range is a run of "units": pieces of query tiles.  A
// query tile wholly inside one range is finished by that CTA as in the plain
// kernel; a tile cut by range boundaries leaves its pieces' unnormalised
// states (row maximum, row sum, output) in the workspace, and the CTA whose
// piece arrives last merges them (log-sum-exp) and writes the tile's output,
// counting arrivals in a per-tile counter that it sets back to zero.
//
// The roles are those of the plain kernel, each looping over the CTA's units
// with its tile counter g running on across units (ring stages, S/P buffers
// and barrier phases follow g): a unit's Q is loaded once the previous unit's
// last QK^T has completed (q_free), and its first P V product waits until the
// previous unit's epilogue has read O out of tensor memory (o_free).  The V
// ring has two stages here, which leaves room for the unit bookkeeping.
// ============================================================================

constexpr int kBVStages = 2;
constexpr int B_OFF_Q = 0;
constexpr int B_OFF_K = 2 * kHalf;
constexpr int B_OFF_V = B_OFF_K + kKStages * 2 * kHalf;
constexpr int B_OFF_X = B_OFF_V + kBVStages * 2 * kHalf;              // (m, l) exchange [unit parity][half][128]
constexpr int B_OFF_PFX = B_OFF_X + 2 * 2 * 128 * 8;                  // pair prefix over chunks [kMax + 1]
constexpr int B_OFF_ROW = B_OFF_PFX + (kMaxChunksBalanced + 1) * 4;   // row prefix over chunks [kMax + 1]
constexpr int B_OFF_MISC = B_OFF_ROW + (kMaxChunksBalanced + 1) * 4;  // scan totals, merge decisions
constexpr int B_OFF_BAR = B_OFF_MISC + 128;
constexpr int B_SMEM_BYTES = B_OFF_BAR + 256 + 1024;
static_assert(B_SMEM_BYTES <= 232448, "shared memory");

struct BBars {
  uint64_t q_full, q_free;
  uint64_t k_full[kKStages], s_full[kKStages];
  uint64_t v_full[kBVStages], p_full[kBVStages], pv_done[kBVStages];
  uint64_t x_full, o_free, drain;
  uint32_t tmem_base;
};
static_assert(sizeof(BBars) <= 256, "barriers");

// Key tiles of one query tile (from its loop's first key tile kt0 to the tile
// holding its last row's last key).
__device__ __forceinline__ int tile_pairs(int start, int ctx, int t0, int TQ, int win) {
  const int last_key = min(start + t0 + TQ - 1, ctx - 1);
  const int klo = (win > 0 && start + t0 - win + 1 > 0) ? start + t0 - win + 1 : 0;
  return last_key / 128 + 1 - klo / 128;
}

__device__ __forceinline__ bool chunk_ok(const PrefillParams &p, int start, int len, int ctx, int row0) {
  return !(len < 1 || len > p.max_chunk_len || start < 0 || ctx != start + len ||
           ctx > p.max_blocks_per_seq * kBlock || row0 + len > p.total_q_tokens);
}

// One unit: key tiles [ka, kb) (counted from kt0) of query tile mt of chunk c, KV head h.
struct Unit {
  int c, h, mt, ka, kb, ntl;
  int start, len, ctx, row0, t0, kt0, pg0, npages, lo_tiles, kt_ctx;
  int64_t tile_off;  // the tile's first pair in the global numbering
};

// The unit that starts at global pair x of a range ending at x_end.  pfx[c]
// counts the pairs of the chunks before c (all KV heads), rows[c] their rows.
template <int G>
__device__ __forceinline__ Unit unit_at(int64_t x, int64_t x_end, const int32_t *pfx, const int32_t *rows,
                                        const PrefillParams &p) {
  constexpr int TQ = 128 / G;
  int lo = 0, hi = p.num_chunks - 1;  // last chunk with pfx[c] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pfx[mid] <= x) lo = mid; else hi = mid - 1;
  }
  Unit u;
  u.c = lo;
  u.start = __ldg(p.chunk_starts + lo);
  u.len = __ldg(p.chunk_lens + lo);
  u.ctx = __ldg(p.context_lens + lo);
  u.row0 = rows[lo];
  const int per_head = (pfx[lo + 1] - pfx[lo]) / p.num_kv_heads;
  int64_t r = x - pfx[lo];
  u.h = (int)(r / per_head);
  r -= (int64_t)u.h * per_head;
  int mt = 0, w = 0;
  for (;; ++mt) {
    w = tile_pairs(u.start, u.ctx, mt * TQ, TQ, p.window);
    if (r < w) break;
    r -= w;
  }
  u.mt = mt;
  u.ntl = w;
  u.ka = (int)r;
  const int64_t rest = x_end - x;
  u.kb = (int64_t)(w - u.ka) < rest ? w : u.ka + (int)rest;
  u.tile_off = x - u.ka;
  u.t0 = mt * TQ;
  const int win = p.window;
  const int klo = (win > 0 && u.start + u.t0 - win + 1 > 0) ? u.start + u.t0 - win + 1 : 0;
  u.kt0 = klo / 128;
  u.pg0 = klo / kBlock;
  u.npages = (u.ctx + kBlock - 1) / kBlock;
  u.lo_tiles = (win > 0 && win < 128) ? w : (u.start + u.t0 < 127 ? 1 : 0);
  u.kt_ctx = (u.ctx - 1) / 128;
  return u;
}

// First pair of CTA b when n CTAs split W pairs as [b W / n, (b + 1) W / n)
// (CTAs b >= n take none), and the CTA owning global pair y.  n is at most W,
// so no range is empty: every CTA between the first and the last owner of a
// tile's pairs holds a piece of it (the merge counts them).
__device__ __forceinline__ int64_t range_start(int b, int64_t W, int n) { return b >= n ? W : (int64_t)b * W / n; }
__device__ __forceinline__ int owner_of(int64_t y, int64_t W, int n) {
  const int64_t b = ((y + 1) * n + W - 1) / W - 1;
  return (int)(b < n - 1 ? b : n - 1);
}

template <typename T, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_balanced_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap qmap, const PrefillParams p) {
  constexpr int TQ = 128 / G;  // query tokens per tile
  constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t IDESC_S = tc::idesc_f16(kBF16, 128, 128, false);
  constexpr uint32_t IDESC_O = tc::idesc_f16(kBF16, 128, 128, true);
  constexpr unsigned FULL = 0xffffffffu;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  BBars &bars = *reinterpret_cast<BBars *>(smem + B_OFF_BAR);
  int32_t *pfx = reinterpret_cast<int32_t *>(smem + B_OFF_PFX);
  int32_t *rows = reinterpret_cast<int32_t *>(smem + B_OFF_ROW);
  int32_t *misc = reinterpret_cast<int32_t *>(smem + B_OFF_MISC);  // [0..15] scan totals, [16..17] merge flags
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = (int)blockIdx.x;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&qmap);
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_free, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars.k_full[i], kLoadWarps);
      mbar_init(&bars.s_full[i], 1);
    }
    for (int i = 0; i < kBVStages; ++i) {
      mbar_init(&bars.v_full[i], kLoadWarps);
      mbar_init(&bars.p_full[i], kSoftmaxThreads);
      mbar_init(&bars.pv_done[i], 1);
    }
    mbar_init(&bars.x_full, kSoftmaxThreads);
    mbar_init(&bars.o_free, kSoftmaxThreads);
    mbar_init(&bars.drain, 1);
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc(&bars.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }

  // ---- the schedule: pairs and rows per chunk, prefix sums (every CTA the same) ----
  // No kernel of this library writes the chunk metadata, so it is read while
  // the previous kernel may still run.  Thread t (t < 256) takes chunk t.
  {
    const int t = threadIdx.x;
    int pairs = 0, len = 0;
    if (t < p.num_chunks) {
      const int start = __ldg(p.chunk_starts + t), ctx = __ldg(p.context_lens + t);
      len = __ldg(p.chunk_lens + t);
      if (len >= 1 && len <= p.max_chunk_len && start >= 0 && ctx == start + len &&
          ctx <= p.max_blocks_per_seq * kBlock) {
        for (int t0 = 0; t0 < len; t0 += TQ) pairs += tile_pairs(start, ctx, t0, TQ, p.window);
        pairs *= p.num_kv_heads;
      }
    }
    // exclusive scans over the first 256 threads (8 warps), pairs and rows together
    int ip = pairs, il = len;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int yp = __shfl_up_sync(FULL, ip, off), yl = __shfl_up_sync(FULL, il, off);
      if (lane >= off) {
        ip += yp;
        il += yl;
      }
    }
    if (lane == 31 && warp < 8) {
      misc[warp] = ip;
      misc[8 + warp] = il;
    }
    __syncthreads();
    if (t < kMaxChunksBalanced) {
      int bp = 0, bl = 0;
      for (int i = 0; i < warp; ++i) {
        bp += misc[i];
        bl += misc[8 + i];
      }
      pfx[t + 1] = bp + ip;
      rows[t + 1] = bl + il;
      if (t == 0) {
        pfx[0] = 0;
        rows[0] = 0;
      }
    }
    __syncthreads();
    // Chunks with inconsistent metadata have no pairs; a chunk whose rows would
    // run past the packed q keeps its pairs but stores nothing.  Both are reported.
    if (b == 0 && t < p.num_chunks && (pairs == 0 || rows[t] + len > p.total_q_tokens))
      set_error(p.err, PA_ERR_RANGE, t);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars.tmem_base;
  const int64_t W = pfx[p.num_chunks];
  const int nb = W < (int64_t)gridDim.x ? (int)W : (int)gridDim.x;  // CTAs with pairs
  const int64_t x0 = range_start(b, W, nb), x1 = range_start(b + 1, W, nb);
  bool timed_out = false;

  if (warp < kSoftmaxWarps) {
    regs_inc<kRegsSoftmax>();
    regs_taken();
    // ---------------- softmax + epilogue (warps 0..7), unit after unit ----------------
    const int quad = warp & 3, ch = warp >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t o_self = tmem + lane_base + kColO + ch * 128;
    const float sl2 = p.scale_log2;
    int g = 0, ui = 0;
    for (int64_t x = x0; x < x1 && !timed_out; ++ui) {
      const Unit U = unit_at<G>(x, x1, pfx, rows, p);
      x += U.kb - U.ka;
      const bool valid = chunk_ok(p, U.start, U.len, U.ctx, U.row0);
      const int tq = U.t0 + r / G;
      const int head = U.h * G + r % G;
      const int lim = min(U.start + tq, U.ctx - 1);
      const int win = p.window;
      const int rlo = (win > 0 && U.start + tq - win + 1 > 0) ? U.start + tq - win + 1 : 0;
      const bool none = lim < rlo;
      const int kb0 = none ? -(1 << 30) : U.kt0 * 128 + ch * 64 - rlo, span = none ? 0 : lim - rlo;
      const int kt_last = U.kt_ctx - U.kt0;
      const int zrow = U.ctx - U.kt_ctx * 128;
      float m_ref = -INFINITY, l = 0.f;

      for (int kt = U.ka; kt < U.kb; ++kt, ++g) {   // kt: tile index from kt0; g: the CTA's tile counter
        const int sb = g & 1, ks = g % kKStages, vs = g % kBVStages;
        if (!mbar_wait(&bars.s_full[ks], (g / kKStages) & 1)) {
          timed_out = true;
          break;
        }
        tc::fence_after_sync();
        const uint32_t s_addr = tmem + lane_base + sb * 128 + ch * 64;
        const int kb = kb0 + kt * 128;
        uint32_t v[2][32];
        tc::ld_32x32b_x32(s_addr, v[0]);
        tc::ld_32x32b_x32(s_addr + 32, v[1]);
        tc::wait_ld();
        const bool full = __all_sync(FULL, kb >= 0 && kb + 63 <= span);
        const bool first = (m_ref == -INFINITY);
        const bool common = kt >= U.lo_tiles && __all_sync(FULL, full && !first);
        float mx = -INFINITY, ls = 0.f;
        if (common) ls = exp_pack_store<T, false>(v, s_addr, sl2, m_ref, true, kb, span);
        if (!common || ls > kRescaleSum) {
          if (full) {
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                float &a = m4[cc * 2 + ((j >> 2) & 1)];
                a = fmax3(a, __uint_as_float(v[cc][j]), __uint_as_float(v[cc][j + 1]));
                a = fmax3(a, __uint_as_float(v[cc][j + 2]), __uint_as_float(v[cc][j + 3]));
              }
            mx = fmaxf(fmax3(m4[0], m4[1], m4[2]), m4[3]);
          } else {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc)
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if ((unsigned)(kb + cc * 32 + j) <= (unsigned)span) mx = fmaxf(mx, __uint_as_float(v[cc][j]));
          }
        }
        const float mc = mx * sl2;
        const bool need = !first && (mc > m_ref + kRescale);
        const bool redo = __any_sync(FULL, need);
        if (redo) {  // warp-uniform; the previous tile (g - 1) belongs to this unit (first is false)
          if (common) tc::wait_st();
          const float f = need ? ex2(m_ref - mc) : 1.f;
          if (need) {
            l *= f;
            m_ref = mc;
          }
          if (!mbar_wait(&bars.pv_done[(g - 1) % kBVStages], ((g - 1) / kBVStages) & 1)) {
            timed_out = true;
            break;
          }
          tc::fence_after_sync();
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t ov[32];
            tc::ld_32x32b_x32(o_self + cc * 32, ov);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
            tc::st_32x32b_x32(o_self + cc * 32, ov);
          }
        }
        if (first) m_ref = mc;
        if (!common || redo) {
          ls = (kt < U.lo_tiles) ? exp_pack_store<T, true>(v, s_addr, sl2, m_ref, full, kb, span)
                                 : exp_pack_store<T, false>(v, s_addr, sl2, m_ref, full, kb, span);
        }
        l += ls;
        tc::wait_st();
        if (kt == kt_last) {  // value rows past the sequence's last key, this half only
          if (!mbar_wait(&bars.v_full[vs], (g / kBVStages) & 1)) {
            timed_out = true;
            break;
          }
          const int z0 = max(zrow, ch * 64), z1 = ch * 64 + 64;
          uint8_t *vbase = smem + B_OFF_V + vs * 2 * kHalf;
          for (int idx = (warp & 3) * 32 + lane; idx < (z1 - z0) * 16; idx += kSoftmaxThreads / 2) {
            const int row = z0 + (idx >> 4), part = idx & 15;
            *reinterpret_cast<uint4 *>(vbase + (row >> 4) * kVPage + (part >> 3) * (kVPage / 2) + (row & 15) * 128 +
                                       (part & 7) * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc::fence_before_sync();
        if (kt != kt_last && !mbar_wait(&bars.v_full[vs], (g / kBVStages) & 1)) {
          timed_out = true;
          break;
        }
        mbar_arrive(&bars.p_full[vs]);
      }
      if (timed_out) break;

      // ---- the unit's epilogue ----
      const int gl = g - 1;  // the unit's last tile
      if (!mbar_wait(&bars.pv_done[gl % kBVStages], (gl / kBVStages) & 1)) {
        timed_out = true;
        break;
      }
      tc::fence_after_sync();
      float2 *xm = reinterpret_cast<float2 *>(smem + B_OFF_X) + (ui & 1) * 256;
      xm[ch * 128 + r] = make_float2(m_ref, l);
      mbar_arrive(&bars.x_full);
      if (!mbar_wait(&bars.x_full, ui & 1)) {
        timed_out = true;
        break;
      }
      const float2 other = xm[(1 - ch) * 128 + r];
      const float m0 = ch == 0 ? m_ref : other.x, l0 = ch == 0 ? l : other.y;
      const float m1 = ch == 0 ? other.x : m_ref, l1 = ch == 0 ? other.y : l;
      const float M = fmaxf(m0, m1);
      const float f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - M);
      const float f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - M);
      const float L = l0 * f0 + l1 * f1;
      // this thread's 64 dims of the row, both key halves, out of tensor memory; then O is free
      const uint32_t o0 = tmem + lane_base + kColO + ch * 64, o1 = o0 + 128;
      uint32_t a[64], bq[64];
      tc::ld_32x32b_x32(o0, *reinterpret_cast<uint32_t(*)[32]>(a));
      tc::ld_32x32b_x32(o0 + 32, *reinterpret_cast<uint32_t(*)[32]>(a + 32));
      tc::ld_32x32b_x32(o1, *reinterpret_cast<uint32_t(*)[32]>(bq));
      tc::ld_32x32b_x32(o1 + 32, *reinterpret_cast<uint32_t(*)[32]>(bq + 32));
      tc::wait_ld();
      tc::fence_before_sync();
      mbar_arrive(&bars.o_free);
      float (&y)[64] = *reinterpret_cast<float(*)[64]>(a);  // the row's unnormalised output, in place
#pragma unroll
      for (int i = 0; i < 64; ++i) y[i] = __uint_as_float(a[i]) * f0 + __uint_as_float(bq[i]) * f1;
      const bool row_ok = valid && tq < U.len;
      T *op = reinterpret_cast<T *>(p.out) + ((int64_t)(U.row0 + tq) * p.num_q_heads + head) * kHeadDim + ch * 64;
      auto store_out = [&](const float (&yy)[64], float inv) {
        if (!row_ok) return;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          uint4 w;
          w.x = Pack<T>::from_f2(yy[8 * i + 0] * inv, yy[8 * i + 1] * inv);
          w.y = Pack<T>::from_f2(yy[8 * i + 2] * inv, yy[8 * i + 3] * inv);
          w.z = Pack<T>::from_f2(yy[8 * i + 4] * inv, yy[8 * i + 5] * inv);
          w.w = Pack<T>::from_f2(yy[8 * i + 6] * inv, yy[8 * i + 7] * inv);
          reinterpret_cast<uint4 *>(op)[i] = w;
        }
      };
      if (U.ka == 0 && U.kb == U.ntl) {
        store_out(y, 1.f / L);
        continue;
      }
      // A piece of a split tile: publish (M, L) and the unnormalised output in
      // this CTA's slot (its first unit: slot 2b, its last: 2b + 1), then count
      // the arrival; the last piece to arrive merges every piece.
      const int slot = 2 * b + (x0 >= U.tile_off ? 0 : 1);
      float *so = p.ws_o + ((int64_t)slot * 128 + r) * kHeadDim + ch * 64;
#pragma unroll
      for (int i = 0; i < 16; ++i)
        reinterpret_cast<float4 *>(so)[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
      if (ch == 0) p.ws_ml[(int64_t)slot * 128 + r] = make_float2(M, L);
      __threadfence();
      named_barrier(2, kSoftmaxThreads);
      const int tile_id = (U.c * p.num_kv_heads + U.h) * p.max_tiles + U.mt;
      const int f_first = owner_of(U.tile_off, W, nb), f_last = owner_of(U.tile_off + U.ntl - 1, W, nb);
      const int nfrag = f_last - f_first + 1;
      if (threadIdx.x == 0) misc[16 + (ui & 1)] = atomicAdd(p.ws_counters + tile_id, 1) == nfrag - 1 ? 1 : 0;
      named_barrier(2, kSoftmaxThreads);
      if (misc[16 + (ui & 1)]) {
        __threadfence();
        float Mx = -INFINITY;
        for (int f = f_first; f <= f_last; ++f) {
          const int sf = 2 * f + (range_start(f, W, nb) >= U.tile_off ? 0 : 1);
          Mx = fmaxf(Mx, __ldcg(p.ws_ml + (int64_t)sf * 128 + r).x);
        }
        float acc[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = 0.f;
        float Ls = 0.f;
        for (int f = f_first; f <= f_last; ++f) {
          const int sf = 2 * f + (range_start(f, W, nb) >= U.tile_off ? 0 : 1);
          const float2 ml = __ldcg(p.ws_ml + (int64_t)sf * 128 + r);
          const float wgt = (ml.x == -INFINITY) ? 0.f : ex2(ml.x - Mx);
          Ls += ml.y * wgt;
          const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + ((int64_t)sf * 128 + r) * kHeadDim + ch * 64);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float4 o4 = __ldcg(src + i);
            acc[4 * i] = fmaf(wgt, o4.x, acc[4 * i]);
            acc[4 * i + 1] = fmaf(wgt, o4.y, acc[4 * i + 1]);
            acc[4 * i + 2] = fmaf(wgt, o4.z, acc[4 * i + 2]);
            acc[4 * i + 3] = fmaf(wgt, o4.w, acc[4 * i + 3]);
          }
        }
        store_out(acc, 1.f / Ls);
        if (threadIdx.x == 0) p.ws_counters[tile_id] = 0;  // ready for the next call
      }
    }
    regs_dec<128>();
  } else {
    // every loader and MMA warp runs this one decrease (setmaxnreg acts on whole warpgroups)
    regs_dec<kRegsOther>();
    if (warp != kWarpMma) {
      // ---------------- loader warps ----------------
      const int lw = warp - kWarpLoad0;
      griddep_wait();  // Q, K and V may come from the previous kernel
      const int kb0 = lw, vb0 = (lw + 5) % kLoadWarps;
      int g = 0, ui = 0, k_issued = 0, v_issued = 0;
      for (int64_t x = x0; x < x1 && !timed_out; ++ui) {
        const Unit U = unit_at<G>(x, x1, pfx, rows, p);
        x += U.kb - U.ka;
        const int32_t *bt = p.block_tables + (int64_t)U.c * p.max_blocks_per_seq;
        if (lw == 0 && lane == 0) {
          if (ui > 0 && !mbar_wait(&bars.q_free, (ui - 1) & 1)) timed_out = true;
          // (rows past the packed q, of a chunk whose rows overrun it, read as zeros; nothing is stored for them)
          mbar_arrive_expect_tx(&bars.q_full, 2 * kHalf);
          tma_load_3d(smem + B_OFF_Q, &qmap, &bars.q_full, 0, U.h * G, U.row0 + U.t0);
          tma_load_3d(smem + B_OFF_Q + kHalf, &qmap, &bars.q_full, 64, U.h * G, U.row0 + U.t0);
        }
        timed_out = __any_sync(FULL, timed_out);
        for (int t = U.ka; t < U.kb && !timed_out; ++t, ++g) {
          const int ks = g % kKStages, vs = g % kBVStages;
          if (g >= kKStages && !mbar_wait(&bars.s_full[ks], ((g - kKStages) / kKStages) & 1)) {
            timed_out = true;
            break;
          }
          load_boxes(smem + B_OFF_K + ks * 2 * kHalf, &kmap, &bars.k_full[ks], U.kt0 + t, kb0, U.h, U.pg0, U.npages,
                     nullptr, bt, p, U.c, lane);
          k_issued = g + 1;
          if (g >= kBVStages && !mbar_wait(&bars.pv_done[vs], ((g - kBVStages) / kBVStages) & 1)) {
            timed_out = true;
            break;
          }
          load_vpages(smem + B_OFF_V + vs * 2 * kHalf, &vmap, &bars.v_full[vs], U.kt0 + t, vb0, U.h, U.pg0,
                      U.npages, nullptr, bt, p, U.c, lane);
          v_issued = g + 1;
        }
      }
      if (timed_out) {  // a short, bounded chance for this warp's copies in flight to land
        for (int t = k_issued - kKStages > 0 ? k_issued - kKStages : 0; t < k_issued; ++t)
          mbar_wait(&bars.k_full[t % kKStages], (t / kKStages) & 1, kWaitLimitNs / 8);
        for (int t = v_issued - kBVStages > 0 ? v_issued - kBVStages : 0; t < v_issued; ++t)
          mbar_wait(&bars.v_full[t % kBVStages], (t / kBVStages) & 1, kWaitLimitNs / 8);
      }
    } else {
      // ---------------- MMA issuer (warp-uniform loop, one elected lane issues) ----------------
      const bool leader = elect_one();
      auto wait_all = [&](uint64_t *bar, uint32_t parity) { return __all_sync(FULL, mbar_wait(bar, parity)) != 0; };
      const uint64_t qdesc = tc::desc_sw128(smem_u32(smem + B_OFF_Q), 16, 1024);
      const uint64_t kdesc0 = tc::desc_sw128(smem_u32(smem + B_OFF_K), 16, 1024);
      const uint64_t vdesc0 = tc::desc_sw128(smem_u32(smem + B_OFF_V), kVPage / 2, 1024);
      constexpr uint64_t kStageStep = (2 * kHalf) >> 4;
      constexpr uint64_t kHalfStep = kHalf >> 4;
      // the P V product of tile pg (pending), issued once P is ready
      int pg = -1, p_unit = 0;
      bool p_first = false, p_lo = false;
      auto issue_pv = [&]() -> bool {
        const int jv = pg % kBVStages;
        if (!wait_all(&bars.p_full[jv], (pg / kBVStages) & 1)) return false;
        if (p_first && p_unit > 0 && !wait_all(&bars.o_free, (p_unit - 1) & 1)) return false;
        tc::fence_after_sync();
        const uint64_t vdesc = vdesc0 + (uint64_t)jv * kStageStep;
        const uint32_t p_col = tmem + (pg & 1) * 128;
        const uint32_t acc0 = p_first ? 0u : 1u;
        if (leader) {
          if (p_lo) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t o_col = tmem + kColO + (kk >> 2) * 128;
              const uint32_t a_hi = p_col + 32 * (kk >> 1) + 8 * (kk & 1);
              const uint64_t bdesc = vdesc + (uint64_t)(kk * (kVPage >> 4));
              tc::mma_f16_ts(o_col, a_hi, bdesc, IDESC_O, (kk & 3) > 0 ? 1u : acc0);
              tc::mma_f16_ts(o_col, a_hi + 16, bdesc, IDESC_O, 1u);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t o_col = tmem + kColO + (kk >> 2) * 128;
              const uint32_t a_hi = p_col + 32 * (kk >> 1) + 8 * (kk & 1);
              const uint64_t bdesc = vdesc + (uint64_t)(kk * (kVPage >> 4));
              tc::mma_f16_ts(o_col, a_hi, bdesc, IDESC_O, (kk & 3) > 0 ? 1u : acc0);
            }
          }
          tc::commit(&bars.pv_done[jv]);
        }
        __syncwarp();
        return true;
      };
      int g = 0, ui = 0;
      for (int64_t x = x0; x < x1 && !timed_out; ++ui) {
        const Unit U = unit_at<G>(x, x1, pfx, rows, p);
        x += U.kb - U.ka;
        // the previous unit's last P V first: its epilogue need not wait for this unit's Q and first K
        if (pg >= 0) {
          if (!issue_pv()) {
            timed_out = true;
            break;
          }
          pg = -1;
        }
        if (!wait_all(&bars.q_full, ui & 1)) {
          timed_out = true;
          break;
        }
        for (int kt = U.ka; kt < U.kb; ++kt, ++g) {
          const int ks = g % kKStages;
          if (!wait_all(&bars.k_full[ks], (g / kKStages) & 1)) {
            timed_out = true;
            break;
          }
          tc::fence_after_sync();
          const uint64_t kdesc = kdesc0 + (uint64_t)ks * kStageStep;
          const uint32_t s_col = tmem + (g & 1) * 128;
          if (leader) {
            tc::mma_f16(s_col, qdesc, kdesc, IDESC_S, 0u);
#pragma unroll
            for (int kk = 1; kk < 8; ++kk) {
              const uint64_t off = (uint64_t)((kk >> 2) * kHalfStep + (kk & 3) * 2);
              tc::mma_f16(s_col, qdesc + off, kdesc + off, IDESC_S, 1u);
            }
            tc::commit(&bars.s_full[ks]);
            if (kt == U.kb - 1) tc::commit(&bars.q_free);  // the unit's Q is no longer read
          }
          __syncwarp();
          if (pg >= 0 && !issue_pv()) {
            timed_out = true;
            break;
          }
          pg = g;
          p_unit = ui;
          p_first = (kt == U.ka);
          p_lo = kt < U.lo_tiles;
        }
      }
      if (!timed_out && pg >= 0 && !issue_pv()) timed_out = true;
      if (timed_out) {
        if (leader) tc::commit(&bars.drain);
        __syncwarp();
        mbar_wait(&bars.drain, 0, kWaitLimitNs / 8);
      }
    }
    regs_wait_taken();  // (the softmax warps hold their registers by now)
    regs_inc<128>();
  }
  if (timed_out) set_error(p.err, PA_ERR_TIMEOUT, b);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  griddep_launch_dependents();
}

template <typename T, int G>
cudaError_t launch_typed(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                         const CUtensorMap &qmap, const CUtensorMap &omap, cudaStream_t stream) {
  if (p.ws_counters) {  // balanced: one CTA per SM
    static KernelSetup bsetup;
    cudaError_t e = kernel_setup(bsetup, prefill_balanced_kernel<T, G>, B_SMEM_BYTES, kThreads, nullptr);
    if (e != cudaSuccess) return e;
    return launch_pdl(prefill_balanced_kernel<T, G>, dim3(sm_count()), dim3(kThreads), B_SMEM_BYTES, stream, kmap,
                      vmap, qmap, p);
  }
  static KernelSetup setup;
  cudaError_t e = kernel_setup(setup, prefill_kernel<T, G>, SMEM_BYTES, kThreads, nullptr);
  if (e != cudaSuccess) return e;
  constexpr int TQ = 128 / G;
  dim3 grid((p.max_chunk_len + TQ - 1) / TQ, p.num_kv_heads, p.num_chunks);
  return launch_pdl(prefill_kernel<T, G>, grid, dim3(kThreads), SMEM_BYTES, stream, kmap, vmap, qmap, omap, p);
}

}  // namespace

// counters [num_chunks][Hkv][max_tiles] int32, then per partial slot (two per
// CTA) 128 rows of (max, sum) and 128 rows of 128 fp32 outputs
size_t prefill_workspace_bytes(int num_chunks, int num_q_heads, int num_kv_heads, int max_chunk_len, int sms) {
  if (num_chunks < 1 || num_kv_heads < 1 || num_q_heads < num_kv_heads || max_chunk_len < 1 || sms < 1) return 0;
  const int tq = 128 / (num_q_heads / num_kv_heads);
  const size_t tiles = (size_t)num_chunks * num_kv_heads * ((max_chunk_len + tq - 1) / tq);
  const size_t counters = (tiles * 4 + 255) & ~(size_t)255;
  const size_t slots = 2 * (size_t)sms;
  return counters + slots * 128 * sizeof(float2) + slots * 128 * kHeadDim * sizeof(float);
}

bool prefill_workspace_carve(void *ws, size_t bytes, int num_chunks, int num_q_heads, int num_kv_heads,
                             int max_chunk_len, int sms, PrefillParams &p) {
  const size_t need = prefill_workspace_bytes(num_chunks, num_q_heads, num_kv_heads, max_chunk_len, sms);
  if (need == 0 || bytes < need) return false;
  const int tq = 128 / (num_q_heads / num_kv_heads);
  p.max_tiles = (max_chunk_len + tq - 1) / tq;
  const size_t tiles = (size_t)num_chunks * num_kv_heads * p.max_tiles;
  const size_t counters = (tiles * 4 + 255) & ~(size_t)255;
  uint8_t *b = static_cast<uint8_t *>(ws);
  p.ws_counters = reinterpret_cast<int32_t *>(b);
  p.ws_ml = reinterpret_cast<float2 *>(b + counters);
  p.ws_o = reinterpret_cast<float *>(b + counters + 2 * (size_t)sms * 128 * sizeof(float2));
  return true;
}

cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const CUtensorMap &qmap, const CUtensorMap &omap, int dtype, int group,
                           cudaStream_t stream) {
#define PA_PREFILL_CASE(T, G) \
  if (group == G) return launch_typed<T, G>(p, kmap, vmap, qmap, omap, stream);
  if (dtype == PA_BF16) {
    PA_PREFILL_CASE(__nv_bfloat16, 1)
    PA_PREFILL_CASE(__nv_bfloat16, 2)
    PA_PREFILL_CASE(__nv_bfloat16, 4)
    PA_PREFILL_CASE(__nv_bfloat16, 8)
  } else {
    PA_PREFILL_CASE(__half, 1)
    PA_PREFILL_CASE(__half, 2)
    PA_PREFILL_CASE(__half, 4)
    PA_PREFILL_CASE(__half, 8)
  }
#undef PA_PREFILL_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
