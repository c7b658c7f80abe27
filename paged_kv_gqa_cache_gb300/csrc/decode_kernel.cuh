#pragma once
// Paged GQA decode for sm_103a: one 2-CTA cluster per (sequence, KV head) when
// those fit on the SMs, else split-K over balanced page ranges plus a combine.
//
// Computes, for every sequence s and query head g (page "Модуль 12: Финальный
// проект: мини-движок инференса", qwen_serve/model.py, Qwen3Model.forward with
// one new token; page "Модуль 04: KV-кэш и арифметика памяти", section 1):
//     out[s][g] = softmax_j(scale * q[s][g] . K_j) V_j,   j < context_lens[s],
// with K_j, V_j taken from KV head g / G of logical position j, which lives in
// block block_tables[s][j / 16] at in-block offset j % 16.  With a sliding
// window of W keys (same page, sections 4 and 5.2) only j >= context_lens[s] - W
// are visible, and pages wholly before the window are never read.
//
// Work decomposition.  The unit of work is one 16-token page of one KV head
// of one sequence ("page" below); a (sequence, KV head) pair is an "item".
// Pages are numbered globally, sequence-major then KV head then page, and the
// W warps of the launch each take one contiguous, equal-sized range of that
// numbering (stream-K style), so every warp moves the same number of bytes
// whatever the length mix.  A warp whose range covers a whole item writes the
// final output itself; otherwise each piece ("fragment") of an item writes an
// unnormalised partial (m, l, o) into slot item + warp of the workspace, and
// the combine kernel merges the fragments of each item with log-sum-exp
// weights.  Every CTA recomputes the per-sequence page prefix sums from
// context_lens, so no planning pass or atomic counter is needed.
//
// Per warp, K/V pages stream through a ring of shared-memory stages filled by
// TMA (one 4-D tensor map per pool; one 4 KB box {128 dims, 1 head, 16 slots}
// per page of K and one of V: the TMA engine's cost grows with the number of
// boxes, so a page is never split) and guarded by one mbarrier each.  One page of K feeds all G query
// heads of its KV head: the scores for G heads come from a single read of K.
// The arithmetic runs on the CUDA cores (fp32; exact int32 dot products for the
// keys of an int8 pool): decode reads each K/V byte once and does G
// multiply-adds per element, far below the tensor-core ridge point.
//
// The one-cluster path (decode_item_kernel) gives each (sequence, KV head) its
// own 16 warps, interleaving its pages over them; the two CTAs merge their
// warps in shared memory and then through the cluster, with no workspace and
// no second launch.
//
// Options: an int8 pool (codes with per-token scales; "Модуль 04", section 5),
// a sliding window, and the KV write of each sequence's new token fused into
// the page that holds it.
#include <type_traits>

#include "pa_device.cuh"

namespace pa {
namespace {

constexpr int NW = kDecodeWarps;
constexpr int STAGE = kDecodeStageBytes;
constexpr int kStages = 3;  // TMA stages per warp
constexpr unsigned FULL = 0xffffffffu;

// Lane layout of the score (QK) phase: NQ adjacent lanes split the 128 dims of
// one key (lane = key * NQ + qd), NT keys are scored per pass, NP passes cover a
// 16-token page.  Lane qd owns the 16-byte chunks qd + NQ * k (k < CPL) of a
// key row; on iteration i it reads chunk qd + NQ * ((i + key) % CPL), so the
// NQ lanes of one key and those of the next key hit disjoint banks of the
// unswizzled 256-byte rows (an 8-lane shared-memory phase covers all 32 banks).
template <int G>
struct Layout {
  static constexpr int NQ = (G >= 8) ? 8 : 4;
  static constexpr int NT = 32 / NQ;
  static constexpr int NP = 16 / NT;
  static constexpr int DPL = 128 / NQ;  // dims per lane
  static constexpr int CPL = DPL / 8;   // 16-byte chunks per lane
};

// First key position a sequence of length ctx attends to: with a sliding
// window of W keys ("Модуль 04: KV-кэш и арифметика памяти", sections 4 and
// 5.2) only the last W positions, else all.  Pages wholly before it are never
// read (their table entries may already be freed).
__device__ __forceinline__ int window_lo(int ctx, int window) { return window > 0 && ctx > window ? ctx - window : 0; }

// Pages of sequence s that hold visible keys (from its window's first page).
__device__ __forceinline__ int pages_of(const DecodeParams &p, int s, bool report) {
  const int ctx = __ldg(p.context_lens + s);
  if (ctx < 1 || ctx > p.max_blocks_per_seq * kBlock) {
    if (report) set_error(p.err, PA_ERR_RANGE, s);
    return 0;
  }
  return (ctx + kBlock - 1) / kBlock - window_lo(ctx, p.window) / kBlock;
}

// Exclusive prefix of pages over sequences into prefix[0..S]: all NT threads
// of the CTA (warp_tot: NT / 32 ints of shared memory); bad lengths are
// reported when `report`.
template <int NT>
__device__ void scan_pages_n(const DecodeParams &p, int32_t *prefix, int *warp_tot, bool report) {
  constexpr int NWT = NT / 32;
  const int n = p.num_seqs;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + NT - 1) / NT;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int sum = 0;
  for (int s = lo; s < hi; ++s) sum += pages_of(p, s, report);
  int incl = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(FULL, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  int base = 0, total = 0;
#pragma unroll
  for (int i = 0; i < NWT; ++i) {
    base += (i < warp) ? warp_tot[i] : 0;
    total += warp_tot[i];
  }
  int run = base + incl - sum;
  for (int s = lo; s < hi; ++s) {
    prefix[s] = run;
    run += pages_of(p, s, false);
  }
  if (tid == 0) prefix[n] = total;
  __syncthreads();
}
__device__ __forceinline__ void scan_pages(const DecodeParams &p, int32_t *prefix, int *warp_tot) {
  scan_pages_n<NW * 32>(p, prefix, warp_tot, blockIdx.x == 0);
}

struct Cursor {
  int s, h, page, pages;
};

__device__ __forceinline__ Cursor locate(const int32_t *prefix, int n, int hkv, int64_t x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)hkv * prefix[mid] <= x) lo = mid; else hi = mid - 1;
  }
  Cursor c;
  c.s = lo;
  c.pages = prefix[lo + 1] - prefix[lo];
  const int64_t r = x - (int64_t)hkv * prefix[lo];
  c.h = (int)(r / c.pages);
  c.page = (int)(r % c.pages);
  return c;
}

__device__ __forceinline__ void advance(Cursor &c, const int32_t *prefix, int n, int hkv) {
  if (++c.page < c.pages) return;
  c.page = 0;
  if (++c.h < hkv) return;
  c.h = 0;
  do {
    ++c.s;
  } while (c.s < n && prefix[c.s + 1] == prefix[c.s]);
  c.pages = (c.s < n) ? prefix[c.s + 1] - prefix[c.s] : 1;
}

// A stage holds one page of one KV head.  16-bit pools: K rows (256 B) at 0,
// V rows at 4096.  int8 pools ("Модуль 04: KV-кэш и арифметика памяти",
// section 5, KV8Cache: one fp32 scale per token and KV head): K codes (128 B
// rows) at 0, V codes at 2048, the page's 16 K scales at 4096 and 16 V scales
// at 4160.
constexpr int kQ8V = 2048, kQ8KS = 4096, kQ8VS = 4160, kQ8StageBytes = 4224;
static_assert(kQ8StageBytes <= STAGE, "an int8 page fits a stage");
// Stage stride in shared memory: a 16-bit page takes 8 KB, an int8 page (codes
// and scales) 4224 bytes, rounded up to the 128-byte alignment of a tensor copy.
template <bool Q8>
__host__ __device__ constexpr int stage_stride() {
  return Q8 ? (kQ8StageBytes + 127) / 128 * 128 : STAGE;
}

// Fetch page blk of KV head h into the stage at dst, completing on bar.
template <bool Q8>
__device__ __forceinline__ void load_page(uint8_t *dst, const CUtensorMap *kmap, const CUtensorMap *vmap,
                                          uint64_t *bar, const DecodeParams &p, int h, int blk) {
  if constexpr (Q8) {
    mbar_arrive_expect_tx(bar, kQ8StageBytes);
    tma_load_4d(dst, kmap, bar, 0, h, 0, blk);
    tma_load_4d(dst + kQ8V, vmap, bar, 0, h, 0, blk);
    const int64_t si = ((int64_t)blk * p.num_kv_heads + h) * kBlock;  // scales of (block, head): 64 B
    bulk_load(dst + kQ8KS, p.k_scale + si, kBlock * 4, bar);
    bulk_load(dst + kQ8VS, p.v_scale + si, kBlock * 4, bar);
  } else {
    mbar_arrive_expect_tx(bar, STAGE);
    tma_load_4d(dst, kmap, bar, 0, h, 0, blk);
    tma_load_4d(dst + 4096, vmap, bar, 0, h, 0, blk);
  }
}

// This lane's dims of the G query rows.  16-bit pools: fp32 pairs pre-scaled
// into the log2 domain.  int8 pools: the row quantised to int16 with one fp32
// scale per row (|error| <= scale / 2, scale = max |q| / 32767, far below the
// 16-bit input's own resolution for every element within 2^7 of the row's
// maximum), so that a key's dot product is exact integer arithmetic on its
// int8 codes (dp2a: two int16 x int8 products per instruction, no code
// conversion) and costs half the registers.
template <bool Q8>
using QReg = typename std::conditional<Q8, uint32_t, float2>::type;

template <typename T, int G, bool Q8>
__device__ __forceinline__ void load_q(const T *qp, float scale_log2, int lane, QReg<Q8> (&q)[G][Layout<G>::DPL / 2],
                                       float (&qsc)[G]) {
  using Ly = Layout<G>;
  constexpr int NQ = Ly::NQ, CPL = Ly::CPL;
  const int qd = lane % NQ, rot = (lane / NQ) % CPL;
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    float2 f[Ly::DPL / 2];
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int chunk = qd + NQ * ((i + rot) % CPL);
      const uint4 u = *reinterpret_cast<const uint4 *>(qp + gg * kHeadDim + chunk * 8);
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) f[i * 4 + e] = Pack<T>::to_f2(wd[e]);
    }
    if constexpr (Q8) {
      float amax = 0.f;
#pragma unroll
      for (int k = 0; k < Ly::DPL / 2; ++k) amax = fmaxf(amax, fmaxf(fabsf(f[k].x), fabsf(f[k].y)));
#pragma unroll
      for (int off = 1; off < NQ; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const float inv = amax > 0.f ? 32767.f / amax : 0.f;
#pragma unroll
      for (int k = 0; k < Ly::DPL / 2; ++k) {
        const int a = __float2int_rn(f[k].x * inv), b = __float2int_rn(f[k].y * inv);
        q[gg][k] = (uint32_t)(a & 0xffff) | ((uint32_t)b << 16);
      }
      qsc[gg] = amax * (1.f / 32767.f) * scale_log2;
    } else {
#pragma unroll
      for (int k = 0; k < Ly::DPL / 2; ++k) q[gg][k] = make_float2(f[k].x * scale_log2, f[k].y * scale_log2);
      qsc[gg] = 1.f;
    }
  }
}

// Append: the new token of sequence s (position ctx - 1, row r of its last
// page, block blk) for KV head h goes into that page's shared-memory stage —
// after the page's copy has landed, so the stage holds the new row whatever
// the copy read there — and into the pool.  One warp; every lane moves 8 of
// the 256 bytes of the K row and of the V row.  The stage is rewritten through
// the generic proxy, so the caller fences before a later copy reuses it.
template <typename T>
__device__ __forceinline__ void append_row(uint8_t *stage, const DecodeParams &p, int s, int h, int blk, int r,
                                           int lane) {
  const int64_t src = ((int64_t)s * p.num_kv_heads + h) * kHeadDim + 4 * lane;
  const uint2 kr = *reinterpret_cast<const uint2 *>(static_cast<const T *>(p.k_new) + src);
  const uint2 vr = *reinterpret_cast<const uint2 *>(static_cast<const T *>(p.v_new) + src);
  *reinterpret_cast<uint2 *>(stage + r * (kHeadDim * 2) + lane * 8) = kr;
  *reinterpret_cast<uint2 *>(stage + kBlock * kHeadDim * 2 + r * (kHeadDim * 2) + lane * 8) = vr;
  const int64_t dst = (((int64_t)blk * kBlock + r) * p.num_kv_heads + h) * kHeadDim + 4 * lane;
  *reinterpret_cast<uint2 *>(static_cast<T *>(p.k_pool) + dst) = kr;
  *reinterpret_cast<uint2 *>(static_cast<T *>(p.v_pool) + dst) = vr;
  __syncwarp();
}

// Scores, online-softmax update and P V of one 16-key page for the G query
// heads of a KV head, from a stage laid out as above (one warp; keys nlo ..
// nv - 1 of the page are visible).  q holds this lane's dims of the G query rows (pre-scaled, log2
// domain); (m, l, o) is the running state (m warp-uniform, l per lane, o for
// the lane's 4 dims).  pbuf2 is the warp's [16 keys][G] scratch for the
// probabilities.  With int8 codes a key's scale multiplies its dot product
// once, and a value's scale multiplies its probability before the sum.
template <typename T, int G, bool Q8, bool F8>
__device__ __forceinline__ void decode_page(const uint8_t *kst, int nlo, int nv,
                                            const QReg<Q8 && !F8> (&q)[G][Layout<G>::DPL / 2], const float (&qsc)[G],
                                            float2 (&o)[G][2], float (&m)[G], float (&l)[G], float2 *pbuf2,
                                            int lane) {
  using Ly = Layout<G>;
  constexpr int NQ = Ly::NQ, NT = Ly::NT, NP = Ly::NP, CPL = Ly::CPL;
  const int qd = lane % NQ;  // which dim slice of a key this lane scores
  const int tk = lane / NQ;  // which key of a pass
  const int rot = tk % CPL;  // chunk rotation of this lane's keys (NT is a multiple of CPL)
  const float neg_inf = -INFINITY;
  const uint8_t *vst = kst + (Q8 ? kQ8V : 4096);
  const float *kscale = reinterpret_cast<const float *>(kst + kQ8KS);
  const float *vscale = reinterpret_cast<const float *>(kst + kQ8VS);

  // scores: NP passes of NT keys; lanes of one key hold slices of its dims
  float sc[NP][G];
#pragma unroll
  for (int ps = 0; ps < NP; ++ps) {
    const int t = ps * NT + tk;
    float2 acc[G];
    int iacc[G];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      acc[gg] = make_float2(0.f, 0.f);
      iacc[gg] = 0;
    }
#pragma unroll
    for (int i = 0; i < CPL; ++i) {
      const int chunk = qd + NQ * ((i + rot) % CPL);  // dims 8 chunk .. 8 chunk + 7
      if constexpr (F8) {  // E4M3 codes to fp32 (exact), then as the 16-bit path
        const uint2 u = *reinterpret_cast<const uint2 *>(kst + t * 128 + chunk * 8);
        const float2 k2[4] = {e4m3x2_to_f2<0>(u.x), e4m3x2_to_f2<1>(u.x), e4m3x2_to_f2<0>(u.y), e4m3x2_to_f2<1>(u.y)};
#pragma unroll
        for (int e = 0; e < 4; ++e)
#pragma unroll
          for (int gg = 0; gg < G; ++gg) acc[gg] = __ffma2_rn(q[gg][i * 4 + e], k2[e], acc[gg]);
      } else if constexpr (Q8) {
        const uint2 u = *reinterpret_cast<const uint2 *>(kst + t * 128 + chunk * 8);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {  // int16 query pairs x int8 codes, exact in int32
          iacc[gg] = __dp2a_lo((int)q[gg][i * 4 + 0], (int)u.x, iacc[gg]);
          iacc[gg] = __dp2a_hi((int)q[gg][i * 4 + 1], (int)u.x, iacc[gg]);
          iacc[gg] = __dp2a_lo((int)q[gg][i * 4 + 2], (int)u.y, iacc[gg]);
          iacc[gg] = __dp2a_hi((int)q[gg][i * 4 + 3], (int)u.y, iacc[gg]);
        }
      } else {
        const uint4 u = *reinterpret_cast<const uint4 *>(kst + t * 256 + chunk * 16);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 k2 = Pack<T>::to_f2(wd[e]);
#pragma unroll
          for (int gg = 0; gg < G; ++gg) acc[gg] = __ffma2_rn(q[gg][i * 4 + e], k2, acc[gg]);
        }
      }
    }
    const float ksc = Q8 ? kscale[t] : 1.f;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      float a;
      if constexpr (Q8 && !F8) {
        int ia = iacc[gg];  // |partial| < 2^31: 128 products of at most 2^15 x 2^7
#pragma unroll
        for (int off = 1; off < NQ; off <<= 1) ia += __shfl_xor_sync(FULL, ia, off);
        a = (float)ia * (qsc[gg] * ksc);
      } else {
        a = acc[gg].x + acc[gg].y;
#pragma unroll
        for (int off = 1; off < NQ; off <<= 1) a += __shfl_xor_sync(FULL, a, off);
        if constexpr (F8) a *= ksc;
      }
      sc[ps][gg] = (t >= nlo && t < nv) ? a : neg_inf;
    }
  }

  // online softmax update (log2 domain)
#pragma unroll
  for (int gg = 0; gg < G; ++gg) {
    float mp = sc[0][gg];
#pragma unroll
    for (int ps = 1; ps < NP; ++ps) mp = fmaxf(mp, sc[ps][gg]);
#pragma unroll
    for (int off = NQ; off < 32; off <<= 1) mp = fmaxf(mp, __shfl_xor_sync(FULL, mp, off));
    const float mn = fmaxf(m[gg], mp);
    const float alpha = exp2f(m[gg] - mn);
    m[gg] = mn;
    float ls = 0.f;
#pragma unroll
    for (int ps = 0; ps < NP; ++ps) {
      const float pr = exp2f(sc[ps][gg] - mn);
      ls += pr;
      const float pv = Q8 ? pr * vscale[ps * NT + tk] : pr;  // the value's scale rides on its weight
      if (qd == 0) pbuf2[(ps * NT + tk) * G + gg] = make_float2(pv, pv);
    }
    l[gg] = l[gg] * alpha + ls;
    const float2 a2 = make_float2(alpha, alpha);
    o[gg][0] = __fmul2_rn(o[gg][0], a2);
    o[gg][1] = __fmul2_rn(o[gg][1], a2);
  }
  __syncwarp();

  // weighted sum of values: this lane owns dims [4 * lane, 4 * lane + 4)
  auto pv_token = [&](int t) {
    float2 v01, v23;
    if constexpr (F8) {
      const uint32_t w = *reinterpret_cast<const uint32_t *>(vst + t * 128 + 4 * lane);
      v01 = e4m3x2_to_f2<0>(w);
      v23 = e4m3x2_to_f2<1>(w);
    } else if constexpr (Q8) {
      const uint32_t w = *reinterpret_cast<const uint32_t *>(vst + t * 128 + 4 * lane);
      v01 = s8x2_to_f2<0>(w);
      v23 = s8x2_to_f2<1>(w);
    } else {
      const uint2 u = *reinterpret_cast<const uint2 *>(vst + t * 256 + 8 * lane);
      v01 = Pack<T>::to_f2(u.x);
      v23 = Pack<T>::to_f2(u.y);
    }
    float2 pp[G];
    if constexpr (G == 1) {
      pp[0] = pbuf2[t];
    } else {
#pragma unroll
      for (int gg = 0; gg < G; gg += 2) {
        const float4 x = *reinterpret_cast<const float4 *>(pbuf2 + t * G + gg);
        pp[gg] = make_float2(x.x, x.y);
        pp[gg + 1] = make_float2(x.z, x.w);
      }
    }
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      o[gg][0] = __ffma2_rn(pp[gg], v01, o[gg][0]);
      o[gg][1] = __ffma2_rn(pp[gg], v23, o[gg][1]);
    }
  };
  if (nlo == 0 && nv == kBlock) {
#pragma unroll
    for (int t = 0; t < kBlock; ++t) pv_token(t);
  } else {
    for (int t = nlo; t < nv; ++t) pv_token(t);
  }
}

// ---- 8-bit pools on the tensor cores ---------------------------------------
// The split kernel scores int8 / E4M3 pages with mma.sync (m16n8k16, fp16
// operands, fp32 accumulators): decode's arithmetic is tiny next to its bytes,
// but per code the CUDA-core path needs a conversion and G multiply-adds,
// where one packed conversion (E4M3 -> fp16 pair, or int8 -> fp16 pair by a
// byte permute, the offset removed once per score or output, see Mma8)
// feeds the tensor core directly.
//   S = Q K^T   rows = the G query heads (rows G .. 15 zero), columns = the
//               16 keys of the page (two n-tiles of 8), k = the 128 dims, in
//               an order of our choosing: lane (g, t) = (lane / 4, lane % 4)
//               takes dims 32 t + 4 ks .. 32 t + 4 ks + 3 at k-step ks, so
//               its K operand is 32 contiguous code bytes of key row g.
//               Every fp16 product is exact and Q is the 16-bit input times a
//               power of two (exact while above 2^-14 of its row maximum).
//   P           the C fragment of S (lane (g, t): head g, keys 2t, 2t + 1,
//               2t + 8, 2t + 9) is exactly the B fragment the P V product
//               needs, so P never leaves the registers.  A value's scale
//               rides on its weight: P'' = P v_scale / R in fp16, with R a
//               power of two per (sequence, KV head) that moves up (and
//               rescales the accumulators) whenever a page's largest value
//               scale exceeds R 2^12, so P'' stays far from fp16 overflow.
//   O^T += V^T P''^T   rows = dims (m-tile mt, row g -> dim 16 g + 2 mt,
//               row g + 8 -> dim 16 g + 2 mt + 1), columns = heads, k = the
//               16 keys: lane (g, t) permutes the bytes of keys 2t, 2t + 1,
//               2t + 8, 2t + 9 at its 16 dims 16 g .. 16 g + 15 into pairs.
// At the end of an item lane (g, t) holds heads 2t and 2t + 1 (those below
// G) at dims 16 g .. 16 g + 15.
// int8 codes enter both products biased, as c + 1152 (the byte permute
// alone, without the subtraction).  Q K^T then carries 1152 times the query
// row's sum (subtracted from every score), P V 1152 times the sum of the
// fp16 weights P'' (ps tracks it, in the same units and with the same
// rescaling as acc, and the epilogue subtracts it).  |c| <= 127, so the bias
// is at most 9 times the terms it rides on: the fp32 accumulators keep a
// score to about 2^-17 of the largest score the row's norm allows (the int16
// query quantisation of a CUDA-core dot product would give 2^-16), an output
// to about 2^-21 of its weights' sum.
struct Mma8 {
  float acc[8][4];  // O^T fragments, in units of R
  float m, l;       // head lane / 4: running maximum (log2 domain), sum of P over this lane's keys
  float ps;         // int8: sum of this lane's P'' (fp16 values as multiplied), head lane / 4
  float R;          // the item's value-scale unit (a power of two; 0 before the first page)
};
constexpr float kQ8Bias = 1152.f;

// (no side effects beyond its outputs: not volatile, so independent products can be interleaved)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// E4M3 codes 0, 1 (I = 0) or 2, 3 (I = 1) of the word w as an fp16 pair,
// exactly: the hardware conversion of one 16-bit half of w (code 2I into
// the low fp16).
template <int I>
__device__ __forceinline__ uint32_t e4m3_h2(uint32_t w) {
  uint32_t r;
  if constexpr (I == 0)
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(w));
  else
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}" : "=r"(r) : "r"(w));
  return r;
}

// int8 codes 0, 1 (I = 0) or 2, 3 (I = 1) of w as fp16 pairs c + 1152, exactly.
template <int I>
__device__ __forceinline__ uint32_t codes_h2_biased(uint32_t w) {
  return __byte_perm(w ^ 0x80808080u, 0x64646464u, I ? 0x4342u : 0x4140u);
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// The G query rows as the A operand (lane (g, t): head g, dims 32 t .. 32 t +
// 31, k-step ks in qa[ks]), times 2^e so that the row's largest magnitude
// lies in [2^14, 2^15); qsc = scale_log2 2^-e.
template <typename T, int G>
__device__ __forceinline__ void load_q_mma(const T *qp, float scale_log2, int lane, uint32_t (&qa)[8][2],
                                           float &qsc, float &qbias) {
  const int g = lane >> 2, t = lane & 3;
  float f[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) f[i] = 0.f;
  if (g < G) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 u = *reinterpret_cast<const uint4 *>(qp + g * kHeadDim + t * 32 + i * 8);
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 v = Pack<T>::to_f2(wd[e]);
        f[i * 8 + 2 * e] = v.x;
        f[i * 8 + 2 * e + 1] = v.y;
      }
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(f[i]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  // e = 14 - floor(log2 amax), kept where 2^e and 2^-e are normal fp32 numbers
  int e = amax > 0.f ? 14 - (int)((__float_as_uint(amax) >> 23) & 0xff) + 127 : 0;
  e = max(-120, min(120, e));
  const float sc = __uint_as_float((uint32_t)(127 + e) << 23);
  qsc = scale_log2 * __uint_as_float((uint32_t)(127 - e) << 23);
  float qs = 0.f;  // the row's sum as the product sees it (the fp16 values)
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    qa[ks][0] = pack_h2(f[4 * ks] * sc, f[4 * ks + 1] * sc);
    qa[ks][1] = pack_h2(f[4 * ks + 2] * sc, f[4 * ks + 3] * sc);
    const float2 x = __half22float2(*reinterpret_cast<const __half2 *>(&qa[ks][0]));
    const float2 y = __half22float2(*reinterpret_cast<const __half2 *>(&qa[ks][1]));
    qs += (x.x + x.y) + (y.x + y.y);
  }
  qs += __shfl_xor_sync(0xffffffffu, qs, 1);
  qs += __shfl_xor_sync(0xffffffffu, qs, 2);
  qbias = kQ8Bias * qs;
}

// One 16-key page of an 8-bit pool (stage layout as load_page<true>): the
// scores, the online-softmax update and O^T += V^T P''^T; keys nlo .. nv - 1
// are visible.
template <int G, bool F8>
__device__ __forceinline__ void decode_page_mma(const uint8_t *kst, int nlo, int nv, const uint32_t (&qa)[8][2],
                                                float qsc, float qbias, Mma8 &st, int lane) {
  const int g = lane >> 2, t = lane & 3;
  const uint8_t *vst = kst + kQ8V;
  const float *kscale = reinterpret_cast<const float *>(kst + kQ8KS);
  const float *vscale = reinterpret_cast<const float *>(kst + kQ8VS);

  // S: this lane's scores of head g for keys 2t, 2t + 1 (n-tile 0) and 2t + 8, 2t + 9 (n-tile 1);
  // four independent accumulation chains (n-tile x even / odd k-step)
  uint32_t kw[2][8];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const uint4 *krow = reinterpret_cast<const uint4 *>(kst + (nt * 8 + g) * kHeadDim + t * 32);
    const uint4 k0 = krow[0], k1 = krow[1];
    kw[nt][0] = k0.x; kw[nt][1] = k0.y; kw[nt][2] = k0.z; kw[nt][3] = k0.w;
    kw[nt][4] = k1.x; kw[nt][5] = k1.y; kw[nt][6] = k1.z; kw[nt][7] = k1.w;
  }
  float c[2][2][4] = {};
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t a[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t b[2];
      if constexpr (F8) {
        b[0] = e4m3_h2<0>(kw[nt][ks]);
        b[1] = e4m3_h2<1>(kw[nt][ks]);
      } else {
        b[0] = codes_h2_biased<0>(kw[nt][ks]);
        b[1] = codes_h2_biased<1>(kw[nt][ks]);
      }
      mma_16816(c[nt][ks & 1], a, b);
    }
  }
  // (int8 keys entered as c + 1152: the product carries 1152 times the row's sum, qbias)
  float s[4] = {c[0][0][0] + c[0][1][0] - qbias, c[0][0][1] + c[0][1][1] - qbias, c[1][0][0] + c[1][1][0] - qbias,
                c[1][0][1] + c[1][1][1] - qbias};
  const float2 ks01 = *reinterpret_cast<const float2 *>(kscale + 2 * t);
  const float2 ks23 = *reinterpret_cast<const float2 *>(kscale + 8 + 2 * t);
  const float ksc[4] = {ks01.x, ks01.y, ks23.x, ks23.y};
  const bool full = nlo == 0 && nv == kBlock;  // (warp-uniform) every key of the page is visible
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int key = (i >> 1) * 8 + 2 * t + (i & 1);
    s[i] = (full || (key >= nlo && key < nv)) ? s[i] * (qsc * ksc[i]) : -INFINITY;
  }

  // online softmax (log2 domain), head g's quad of lanes
  float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  const float mn = fmaxf(st.m, mx);
  const float base = mn == -INFINITY ? 0.f : mn;  // no visible key yet: every P is 0
  const float alpha = ex2(st.m - base);            // 0 while nothing was accumulated
  float p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) p[i] = ex2(s[i] - base);
  st.l = st.l * alpha + ((p[0] + p[1]) + (p[2] + p[3]));
  st.m = mn;

  // value scales: the page's largest against R
  const float2 vs01 = *reinterpret_cast<const float2 *>(vscale + 2 * t);
  const float2 vs23 = *reinterpret_cast<const float2 *>(vscale + 8 + 2 * t);
  float vmax = fmaxf(fmaxf(vs01.x, vs01.y), fmaxf(vs23.x, vs23.y));
  vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 1));
  vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, 2));  // all 16 keys: the same in every lane
  float rs = 1.f;
  if (vmax > st.R * 4096.f) {
    const float Rn = __uint_as_float((__float_as_uint(vmax) + 0x007fffffu) & 0xff800000u);  // 2^ceil(log2 vmax)
    rs = st.R / Rn;
    st.R = Rn;
  }
  const float invR = __uint_as_float((254u << 23) - __float_as_uint(st.R));  // 1 / R, exact
  // the accumulators hold heads 2t and 2t + 1: their factors come from those heads' quads
  const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t) * rs;
  const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4) * rs;
  if (__any_sync(0xffffffffu, a0 != 1.f || a1 != 1.f)) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      st.acc[mt][0] *= a0;
      st.acc[mt][1] *= a1;
      st.acc[mt][2] *= a0;
      st.acc[mt][3] *= a1;
    }
  }
  uint32_t pb[2] = {pack_h2(p[0] * (vs01.x * invR), p[1] * (vs01.y * invR)),
                    pack_h2(p[2] * (vs23.x * invR), p[3] * (vs23.y * invR))};
  if (g >= G) pb[0] = pb[1] = 0u;
  if constexpr (!F8) {  // the weights as the product sees them, for the bias
    const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&pb[0]));
    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&pb[1]));
    st.ps = st.ps * (alpha * rs) + ((f0.x + f0.y) + (f1.x + f1.y));
  }

  // O^T += V^T P''^T: value rows of keys 2t, 2t + 1, 2t + 8, 2t + 9 at dims 16 g .. 16 g + 15
  uint4 v0 = *reinterpret_cast<const uint4 *>(vst + (2 * t) * kHeadDim + 16 * g);
  uint4 v1 = *reinterpret_cast<const uint4 *>(vst + (2 * t + 1) * kHeadDim + 16 * g);
  uint4 v2 = *reinterpret_cast<const uint4 *>(vst + (2 * t + 8) * kHeadDim + 16 * g);
  uint4 v3 = *reinterpret_cast<const uint4 *>(vst + (2 * t + 9) * kHeadDim + 16 * g);
  if (!full) {  // rows of invisible keys may hold any bytes (an E4M3 NaN): zero them
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    if (2 * t < nlo || 2 * t >= nv) v0 = z;
    if (2 * t + 1 < nlo || 2 * t + 1 >= nv) v1 = z;
    if (2 * t + 8 < nlo || 2 * t + 8 >= nv) v2 = z;
    if (2 * t + 9 < nlo || 2 * t + 9 >= nv) v3 = z;
  }
  const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
  const uint32_t w2[4] = {v2.x, v2.y, v2.z, v2.w}, w3[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    // bytes (key a, key b) at dim 16 g + 2 mt, then at dim 16 g + 2 mt + 1
    const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
    const uint32_t x = __byte_perm(w0[mt >> 1], w1[mt >> 1], sel);
    const uint32_t y = __byte_perm(w2[mt >> 1], w3[mt >> 1], sel);
    uint32_t a[4];
    if constexpr (F8) {
      a[0] = e4m3_h2<0>(x); a[1] = e4m3_h2<1>(x); a[2] = e4m3_h2<0>(y); a[3] = e4m3_h2<1>(y);
    } else {
      a[0] = codes_h2_biased<0>(x); a[1] = codes_h2_biased<1>(x); a[2] = codes_h2_biased<0>(y); a[3] = codes_h2_biased<1>(y);
    }
    mma_16816(st.acc[mt], a, pb);
  }
}

// Warp of the launch whose page range contains global page x, when W warps
// (W <= P) split P pages as [floor(w P / W), floor((w + 1) P / W)).
__device__ __forceinline__ int worker_of(int64_t x, int64_t P, int64_t W) {
  const int64_t w = ((x + 1) * W + P - 1) / P - 1;
  return (int)(w < W - 1 ? w : W - 1);
}

// Log-sum-exp merge of the nf fragments (slots item + wf .. item + wf + nf - 1)
// of query head gg of item (s, h) into its output row; one warp, lane owns
// dims [4 * lane, 4 * lane + 4).  The (m, l) of up to 32 fragments are read at
// once (one per lane); the o partials are then streamed CHUNK at a time with
// independent loads (the combine kernel takes 32; the split kernel, merging
// in place with its query rows still in registers, takes 8).  The partials
// are read from L2 (ld.global.cg): in the fused path they were written by
// other SMs during this kernel.
template <typename T, int G, int CHUNK>
__device__ __forceinline__ void merge_fragments(const DecodeParams &p, int s, int h, int gg, int wf, int nf, int lane) {
  static_assert(32 % CHUNK == 0, "chunks tile a group of 32 fragments");
  const int64_t slot0 = (int64_t)s * p.num_kv_heads + h + wf;
  float M = -INFINITY, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int base = 0; base < nf; base += 32) {
    const int f = base + lane;
    float mf = -INFINITY, lf = 0.f;
    if (f < nf) {
      const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.ws_ml + ((slot0 + f) * G + gg) * 2));
      mf = ml.x;
      lf = ml.y;
    }
    float mc = mf;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mc = fmaxf(mc, __shfl_xor_sync(FULL, mc, off));
    const float Mn = fmaxf(M, mc);
    if (Mn == -INFINITY) continue;  // no valid fragment yet (uniform)
    const float so = exp2f(M - Mn);
    const float wgt = (mf > -INFINITY) ? exp2f(mf - Mn) : 0.f;
    float lw = lf * wgt;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lw += __shfl_xor_sync(FULL, lw, off);
    L = L * so + lw;
    O.x *= so; O.y *= so; O.z *= so; O.w *= so;
    M = Mn;
    const int cnt = min(32, nf - base);
#pragma unroll 1
    for (int c0 = 0; c0 < cnt; c0 += CHUNK) {
      // issue every load of this chunk before using any of them
      float4 ov[CHUNK];
#pragma unroll
      for (int j = 0; j < CHUNK; ++j)
        if (c0 + j < cnt)
          ov[j] = __ldcg(
              reinterpret_cast<const float4 *>(p.ws_o + ((slot0 + base + c0 + j) * G + gg) * kHeadDim + 4 * lane));
#pragma unroll
      for (int j = 0; j < CHUNK; ++j) {
        const float wj = __shfl_sync(FULL, wgt, c0 + j);
        if (c0 + j < cnt && wj > 0.f) {
          O.x = fmaf(wj, ov[j].x, O.x);
          O.y = fmaf(wj, ov[j].y, O.y);
          O.z = fmaf(wj, ov[j].z, O.z);
          O.w = fmaf(wj, ov[j].w, O.w);
        }
      }
    }
  }
  const float inv = 1.f / L;
  T *op = reinterpret_cast<T *>(p.out) + ((int64_t)s * p.num_q_heads + h * G + gg) * kHeadDim + 4 * lane;
  uint2 pk;
  pk.x = Pack<T>::from_f2(O.x * inv, O.y * inv);
  pk.y = Pack<T>::from_f2(O.z * inv, O.w * inv);
  *reinterpret_cast<uint2 *>(op) = pk;
}

// The fused combine's merge of one item, by the fragment that arrived last;
// then the item's counter goes back to zero.
template <typename T, int G>
__device__ __forceinline__ void merge_item_fused(const DecodeParams &p, int s, int h, int item, int wf, int nf,
                                              int lane) {
  __threadfence();  // acquire: the other fragments' partials, published before their arrivals
#pragma unroll 1
  for (int gg = 0; gg < G; ++gg) merge_fragments<T, G, 4>(p, s, h, gg, wf, nf, lane);
  if (lane == 0) p.counters[item] = 0;
}

// Shared memory of NWC split workers: per warp kStages stages, their
// barriers and a score buffer; then the page prefix (num_seqs + 1 ints).
template <bool Q8, int G, int NWC>
struct SplitSmem {
  static constexpr int kStagesOff = 0;
  static constexpr int kBarsOff = NWC * kStages * stage_stride<Q8>();
  static constexpr int kPbufOff = kBarsOff + NWC * kStages * 8;
  static constexpr int kPrefixOff = kPbufOff + NWC * 16 * G * 8;
};

// Split worker w of W: the pages [w P / W, (w + 1) P / W) of the global
// numbering (P pages in all; prefix: the CTA's page prefix over sequences),
// run by one warp whose shared memory is slot `slot` of the NWC-warp layout
// at smem.  Writes the outputs of the items it covers whole and the
// fragments of the others (merged by the last fragment to arrive when the
// workspace has counters).  w < W and W <= P, so the range is not empty.
template <typename T, int G, bool Q8, bool F8, int NWC>
__device__ __forceinline__ void decode_split_worker(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                                    const DecodeParams &p, uint8_t *smem, const int32_t *prefix,
                                                    int slot, int64_t w, int64_t P, int64_t W) {
  using Ly = Layout<G>;
  using Sm = SplitSmem<Q8, G, NWC>;
  constexpr int NQ = Ly::NQ, DPL = Ly::DPL;
  constexpr int SST = stage_stride<Q8>();
  const int lane = threadIdx.x & 31;
  uint8_t *stages = smem + Sm::kStagesOff + slot * kStages * SST;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Sm::kBarsOff) + slot * kStages;
  float *pbuf = reinterpret_cast<float *>(smem + Sm::kPbufOff) + slot * 16 * G * 2;
  const int n = p.num_seqs, hkv = p.num_kv_heads;
  if (lane == 0) {
#pragma unroll
    for (int st = 0; st < kStages; ++st) mbar_init(&bars[st], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const int64_t x0 = w * P / W;
  const int64_t x1 = (w + 1) * P / W;
  const int64_t npages = x1 - x0;

  Cursor ic = locate(prefix, n, hkv, x0);
  Cursor cc = ic;

  // ---- producer (lane 0 issues; all lanes track the cursor) --------------------
  int win_s = -1, win_base = -1, win_first = 0;
  int32_t win = -1;
  uint32_t bad_mask = 0;
  auto issue_at = [&](int st, const Cursor &at) {
    const int base = at.page & ~31;
    if (at.s != win_s || base != win_base) {
      if (at.s != win_s) win_first = p.window > 0 ? window_lo(__ldg(p.context_lens + at.s), p.window) / kBlock : 0;
      win_s = at.s;
      win_base = base;
      const int pg = base + lane;
      win = (pg < at.pages)
                ? __ldg(p.block_tables + (int64_t)at.s * p.max_blocks_per_seq + win_first + pg)
                : -1;
    }
    const int blk = __shfl_sync(FULL, win, at.page & 31);
    const bool ok = (unsigned)blk < (unsigned)p.num_blocks;
    if (lane == 0) {
      if (ok) {
        load_page<Q8>(stages + st * SST, &kmap, &vmap, &bars[st], p, at.h, blk);
      } else {
        set_error(p.err, PA_ERR_RANGE, at.s);
        mbar_arrive(&bars[st]);
      }
    }
    bad_mask = ok ? (bad_mask & ~(1u << st)) : (bad_mask | (1u << st));
  };
  auto issue = [&](int st) {
    issue_at(st, ic);
    advance(ic, prefix, n, hkv);
  };

  const int npre = (int)(npages < kStages ? npages : kStages);
  if (p.early_pages) {
    // The caller guarantees that the kernels still running write no page but
    // each sequence's last visible one: fetch the others now, the last pages
    // after the wait.
    Cursor deferred[kStages];
    uint32_t dmask = 0;
#pragma unroll
    for (int g = 0; g < kStages; ++g) {
      if (g < npre) {
        if (ic.page == ic.pages - 1) {
          deferred[g] = ic;
          dmask |= 1u << g;
          advance(ic, prefix, n, hkv);
        } else {
          issue(g);
        }
      }
    }
    griddep_wait();
#pragma unroll
    for (int g = 0; g < kStages; ++g)
      if ((dmask >> g) & 1u) issue_at(g, deferred[g]);
  } else {
    for (int g = 0; g < npre; ++g) issue(g);
  }
  if (w == 0 && p.meta)  // the combine kernel's copy of the page prefix (after the wait: the
    for (int i = lane; i <= p.num_seqs; i += 32) p.meta[i] = prefix[i];  // previous call may still read it)

  // ---- consumer state ---------------------------------------------------------
  // Packed fp32x2 arithmetic (FFMA2): q and the partial scores pair adjacent
  // dims, the output accumulators pair adjacent dims of one head.
  // 16-bit pools: the CUDA-core page step's state; 8-bit pools: the tensor-core one's
  QReg<false> q[G][DPL / 2];
  float qsc[G];
  float2 o[G][2];
  float m[G], l[G];
  uint32_t qa[8][2];
  float qsc8 = 0.f, qbias8 = 0.f;
  Mma8 st8;
  int ctx = 0, first = 0, lo_in_first = 0;  // first visible page and key of the item
  bool open = false, whole = false;
  const float neg_inf = -INFINITY;
  float2 *pbuf2 = reinterpret_cast<float2 *>(pbuf);  // [16 keys][G] of (p, p)

  for (int64_t g = 0; g < npages; ++g) {
    const int st = (int)(g % kStages);
    if (!open) {
      // new item: load its G query rows (pre-scaled into the log2 domain)
      const T *qp = reinterpret_cast<const T *>(p.q) +
                    ((int64_t)cc.s * p.num_q_heads + (int64_t)cc.h * G) * kHeadDim;
      if constexpr (Q8) {
        load_q_mma<T, G>(qp, p.scale_log2, lane, qa, qsc8, qbias8);
        if constexpr (F8) qbias8 = 0.f;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) st8.acc[mt][0] = st8.acc[mt][1] = st8.acc[mt][2] = st8.acc[mt][3] = 0.f;
        st8.m = neg_inf;
        st8.l = 0.f;
        st8.ps = 0.f;
        st8.R = 0.f;
      } else {
        load_q<T, G, false>(qp, p.scale_log2, lane, q, qsc);
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          m[gg] = neg_inf;
          l[gg] = 0.f;
          o[gg][0] = make_float2(0.f, 0.f);
          o[gg][1] = make_float2(0.f, 0.f);
        }
      }
      ctx = __ldg(p.context_lens + cc.s);
      first = window_lo(ctx, p.window) / kBlock;
      lo_in_first = window_lo(ctx, p.window) - first * kBlock;
      whole = (cc.page == 0);
      open = true;
    }

    if (!mbar_wait(&bars[st], (uint32_t)((g / kStages) & 1))) {
      if (lane == 0) set_error(p.err, PA_ERR_TIMEOUT, cc.s);
      // give the copies still in flight a short, bounded chance to land
      for (int64_t r = g + 1; r < (npages < g + kStages ? npages : g + kStages); ++r)
        mbar_wait(&bars[r % kStages], (uint32_t)((r / kStages) & 1), kWaitLimitNs / 8);
      return;
    }

    bool appended = false;
    if (!((bad_mask >> st) & 1u)) {
      const int nv = min(kBlock, ctx - (first + cc.page) * kBlock);  // keys of the sequence in this page
      if constexpr (!Q8) {
        if (p.k_new && cc.page == cc.pages - 1) {  // the page of the sequence's new token
          const int blk = __ldg(p.block_tables + (int64_t)cc.s * p.max_blocks_per_seq + first + cc.page);
          append_row<T>(stages + st * SST, p, cc.s, cc.h, blk, nv - 1, lane);
          appended = true;
        }
      }
      if constexpr (Q8)
        decode_page_mma<G, F8>(stages + st * SST, cc.page == 0 ? lo_in_first : 0, nv, qa, qsc8, qbias8, st8, lane);
      else
        decode_page<T, G, false, false>(stages + st * SST, cc.page == 0 ? lo_in_first : 0, nv, q, qsc, o, m, l,
                                        pbuf2, lane);
    }
    __syncwarp();  // every lane is done with this stage and with pbuf
    if (appended) fence_proxy_async_smem();  // the generic writes precede the stage's next copy

    if (g + kStages < npages) issue(st);

    const bool last_of_item = (cc.page == cc.pages - 1);
    if (last_of_item || g == npages - 1) {
      const int item = cc.s * hkv + cc.h;
      const bool final_out = whole && last_of_item;
      if constexpr (Q8) {
        // lane (gl, tl) holds heads 2 tl and 2 tl + 1 at dims 16 gl .. 16 gl + 15; a head's (m, l) lives
        // in the quad of lanes 4 head .. 4 head + 3
        const int gl = lane >> 2, tl = lane & 3;
        float lq = st8.l, pq = st8.ps;
        lq += __shfl_xor_sync(FULL, lq, 1);
        lq += __shfl_xor_sync(FULL, lq, 2);
        pq += __shfl_xor_sync(FULL, pq, 1);
        pq += __shfl_xor_sync(FULL, pq, 2);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int hh = 2 * tl + c;
          const float mh = __shfl_sync(FULL, st8.m, (4 * hh) & 31);
          const float lh = __shfl_sync(FULL, lq, (4 * hh) & 31);
          const float bias = F8 ? 0.f : kQ8Bias * __shfl_sync(FULL, pq, (4 * hh) & 31);
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            st8.acc[mt][c] -= bias;
            st8.acc[mt][2 + c] -= bias;
          }
          if (hh < G) {
            if (final_out) {
              const float f = st8.R / lh;
              uint32_t pk[8];
#pragma unroll
              for (int mt = 0; mt < 8; ++mt) pk[mt] = Pack<T>::from_f2(st8.acc[mt][c] * f, st8.acc[mt][2 + c] * f);
              uint4 *op = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.out) +
                                                    ((int64_t)cc.s * p.num_q_heads + cc.h * G + hh) * kHeadDim +
                                                    16 * gl);
              op[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              op[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            } else {
              const int64_t slot = ((int64_t)item + w) * G + hh;
              float4 *dst = reinterpret_cast<float4 *>(p.ws_o + slot * kHeadDim + 16 * gl);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_float4(st8.acc[2 * i][c] * st8.R, st8.acc[2 * i][2 + c] * st8.R,
                                     st8.acc[2 * i + 1][c] * st8.R, st8.acc[2 * i + 1][2 + c] * st8.R);
              if (gl == 0) *reinterpret_cast<float2 *>(p.ws_ml + slot * 2) = make_float2(mh, lh);
            }
          }
        }
      } else {
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        float lt = l[gg];
#pragma unroll
        for (int off = NQ; off < 32; off <<= 1) lt += __shfl_xor_sync(FULL, lt, off);
        if (final_out) {
          const float inv = 1.f / lt;
          T *op = reinterpret_cast<T *>(p.out) +
                  ((int64_t)cc.s * p.num_q_heads + cc.h * G + gg) * kHeadDim + 4 * lane;
          uint2 pk;
          pk.x = Pack<T>::from_f2(o[gg][0].x * inv, o[gg][0].y * inv);
          pk.y = Pack<T>::from_f2(o[gg][1].x * inv, o[gg][1].y * inv);
          *reinterpret_cast<uint2 *>(op) = pk;
        } else {
          const int64_t slot = ((int64_t)item + w) * G + gg;
          *reinterpret_cast<float4 *>(p.ws_o + slot * kHeadDim + 4 * lane) =
              make_float4(o[gg][0].x, o[gg][0].y, o[gg][1].x, o[gg][1].y);
          if (lane == 0) *reinterpret_cast<float2 *>(p.ws_ml + slot * 2) = make_float2(m[gg], lt);
        }
      }
      }
      if (!final_out && p.counters) {
        // Fused combine: publish this fragment (stores, then a device-scope
        // fence, then the arrival); the fragment that arrives last merges all
        // of the item's fragments and sets the counter back to zero, so the
        // counters are zero again when the kernel ends.
        __threadfence();
        __syncwarp();
        int prev = 0;
        if (lane == 0) prev = atomicAdd(p.counters + item, 1);
        prev = __shfl_sync(FULL, prev, 0);
        const int64_t A = (int64_t)hkv * prefix[cc.s] + (int64_t)cc.h * cc.pages;
        const int wf = worker_of(A, P, W), wl = worker_of(A + cc.pages - 1, P, W);
        if (prev == wl - wf) merge_item_fused<T, G>(p, cc.s, cc.h, item, wf, wl - wf + 1, lane);
      }
      open = false;
    }
    advance(cc, prefix, n, hkv);
  }
}

// 8-bit pools (tensor-core page step, small pages): three CTAs per SM;
// 16-bit pools: as many as fit.
template <typename T, int G, bool Q8, bool F8>
__global__ void __launch_bounds__(NW * 32, Q8 ? 3 : 1)
decode_split_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                    const DecodeParams p) {
  using Sm = SplitSmem<Q8, G, NW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ int warp_tot[NW];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t *prefix = reinterpret_cast<int32_t *>(smem + Sm::kPrefixOff);
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  // The lengths and block tables are never written by the kernels this one
  // may overlap (see griddep_wait); with early_pages they are read, and the
  // first pages fetched, before the wait.
  if (!p.early_pages) griddep_wait();
  scan_pages(p, prefix, warp_tot);

  // With fewer pages than warps only the first P warps work, one page each,
  // so every working warp's range is non-empty (the combine relies on it).
  const int64_t P = (int64_t)prefix[p.num_seqs] * p.num_kv_heads;
  const int64_t W = P < p.num_workers ? P : p.num_workers;
  const int w = blockIdx.x * NW + warp;
  if (w >= W) {
    if (p.early_pages) griddep_wait();
    if (blockIdx.x == 0 && warp == 0)  // only when no warp has pages (W = 0)
      for (int i = lane; i <= p.num_seqs; i += 32) p.meta[i] = prefix[i];
    griddep_launch_dependents();
    return;
  }
  decode_split_worker<T, G, Q8, F8, NW>(kmap, vmap, p, smem, prefix, warp, w, P, W);
  griddep_launch_dependents();
}

}  // namespace
}  // namespace pa
