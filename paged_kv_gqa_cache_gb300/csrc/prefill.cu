// Causal chunked-prefill attention over a paged KV cache on the tcgen05
// tensor cores (sm_103a).
//
// For chunk c (start P, n new tokens, context P + n), query token i at
// absolute position P + i and query head g attends to keys 0 .. P + i of KV
// head g / G, read through the chunk's block table (page "Модуль 12:
// Финальный проект: мини-движок инференса", qwen_serve/model.py,
// Qwen3Model.forward with T > 1: mask kpos <= qpos on absolute positions;
// page "Модуль 04: KV-кэш и арифметика памяти", section 3.4: the prefix KV
// lives in the cache between chunks).
//
// One CTA computes one M = 128 tile of query rows for one KV head: 128 / G
// consecutive tokens of the chunk x the G query heads sharing that KV head,
// so every K/V tile it reads serves all G heads.  Row r of the tile is token
// t0 + r / G, head h * G + r % G (the Q tile is one TMA box per 64-dim half).
// The keys stream in tiles of N = 128 (8 pages, each page one TMA box per
// 64-dim half), double-buffered.  Per key tile:
//   S  = Q K^T   tcgen05.mma kind::f16, A and B K-major, fp32 in TMEM (S0/S1)
//   softmax      warps 0-3 (thread r owns TMEM lane r = row r): masked row
//                max, P = exp2(S * scale * log2 e - m), row sums; P is written
//                to shared memory as two terms in the input dtype, P_hi =
//                round(P) and P_lo = round(P - P_hi) (K-major, 128-byte
//                swizzle), so the tensor-core product sees P to ~16 bits
//   O_t = P V    tcgen05.mma P_hi V + P_lo V, B = V tile MN-major, fp32 in
//                TMEM (O0/O1)
//   O  = O * alpha + O_t  accumulated in registers of the softmax threads.
// Warp 4 issues the TMA loads, warp 5 owns TMEM and issues the MMAs (one
// thread each); mbarriers hand tiles between the roles and every wait is
// bounded.  Keys above the diagonal are masked per element on the tiles that
// cross it and never loaded past the tile holding the tile's last query.
// Value rows past the sequence's last key are zeroed in shared memory before
// the PV product so that a zero probability never meets a non-finite value.
#include <type_traits>

#include "tcgen05.cuh"

namespace pa {
namespace {

constexpr int kThreads = 192;
constexpr int kHalf = 16384;                      // 128 rows x 64 elements x 2 bytes
constexpr int OFF_Q = 0;                          // Q: two 64-dim halves
constexpr int OFF_KV = 2 * kHalf;                 // 2 stages of {K lo, K hi, V lo, V hi}
constexpr int STAGE_BYTES = 4 * kHalf;
constexpr int OFF_P = OFF_KV + 2 * STAGE_BYTES;   // P_hi then P_lo, each two 64-key halves
constexpr int OFF_BAR = OFF_P + 4 * kHalf;
constexpr int SMEM_BYTES = OFF_BAR + 128 + 1024;  // + barriers + alignment slack
constexpr uint32_t kTmemCols = 512;               // S0, S1, O0, O1: 128 columns each

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[2];
  uint64_t s_full[2];
  uint64_t s_free[2];
  uint64_t p_full;
  uint64_t pv_done[2];
  uint32_t tmem_base;
};

// o = o * alpha + (the 128 fp32 columns of this thread's TMEM lane at taddr)
__device__ __forceinline__ void accumulate_o(float (&o)[128], uint32_t taddr, float alpha) {
#pragma unroll
  for (int cch = 0; cch < 4; ++cch) {
    uint32_t v[32];
    tc::ld_32x32b_x32(taddr + cch * 32, v);
    tc::wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) o[cch * 32 + j] = fmaf(o[cch * 32 + j], alpha, __uint_as_float(v[j]));
  }
}

template <typename T, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap qmap, const PrefillParams p) {
  constexpr int TQ = 128 / G;  // query tokens per tile
  constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t IDESC_S = tc::idesc_f16(kBF16, 128, 128, false);
  constexpr uint32_t IDESC_O = tc::idesc_f16(kBF16, 128, 128, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars &bars = *reinterpret_cast<Bars *>(smem + OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_wait();

  // Heaviest tiles first: last chunk, last query tile.
  const int c = p.num_chunks - 1 - (int)blockIdx.z;
  const int h = blockIdx.y;
  const int mt = (int)gridDim.x - 1 - (int)blockIdx.x;
  const int start = __ldg(p.chunk_starts + c), len = __ldg(p.chunk_lens + c), ctx = __ldg(p.context_lens + c);
  int row0 = 0;
  for (int i = 0; i < c; ++i) row0 += __ldg(p.chunk_lens + i);
  const bool bad = len < 1 || len > p.max_chunk_len || start < 0 || ctx != start + len ||
                   ctx > p.max_blocks_per_seq * kBlock || row0 + len > p.total_q_tokens;
  if (bad) {
    if (mt == 0 && h == 0 && threadIdx.x == 0) set_error(p.err, PA_ERR_RANGE, c);
    griddep_launch_dependents();
    return;
  }
  const int t0 = mt * TQ;
  if (t0 >= len) {
    griddep_launch_dependents();
    return;
  }
  const int last_key = min(start + t0 + TQ - 1, ctx - 1);  // largest key any row of the tile sees
  const int nkt = last_key / 128 + 1;
  const int kt_ctx = (ctx - 1) / 128;                       // key tile holding the sequence's last key
  const int npages = (ctx + kBlock - 1) / kBlock;
  const int32_t *bt = p.block_tables + (int64_t)c * p.max_blocks_per_seq;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&qmap);
    mbar_init(&bars.q_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.kv_full[b], 1);
      mbar_init(&bars.s_full[b], 1);
      mbar_init(&bars.s_free[b], 128);
      mbar_init(&bars.pv_done[b], 1);
    }
    mbar_init(&bars.p_full, 128);
    fence_mbar_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(&bars.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars.tmem_base;
  bool timed_out = false;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars.q_full, 2 * kHalf);
      tma_load_3d(smem + OFF_Q, &qmap, &bars.q_full, 0, h * G, row0 + t0);
      tma_load_3d(smem + OFF_Q + kHalf, &qmap, &bars.q_full, 64, h * G, row0 + t0);
      for (int kt = 0; kt < nkt; ++kt) {
        const int b = kt & 1;
        if (kt >= 2 && !mbar_wait(&bars.pv_done[b], ((kt - 2) >> 1) & 1)) {
          timed_out = true;
          break;
        }
        uint8_t *st = smem + OFF_KV + b * STAGE_BYTES;
        const int pg0 = kt * 8;
        const int np = min(8, npages - pg0);
        int blk[8];
        int nvalid = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          blk[j] = -1;
          if (j < np) {
            const int id = __ldg(bt + pg0 + j);
            if ((unsigned)id < (unsigned)p.num_blocks) {
              blk[j] = id;
              ++nvalid;
            } else {
              set_error(p.err, PA_ERR_RANGE, c);
            }
          }
        }
        // A page whose block id is out of range is not loaded; zero it so the
        // products stay finite (the error word already reports the chunk).
        bool zeroed = false;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (j >= np || blk[j] >= 0) continue;
          for (int part = 0; part < 4; ++part) {
            uint4 *z = reinterpret_cast<uint4 *>(st + part * kHalf + j * 2048);
            for (int i = 0; i < 128; ++i) z[i] = make_uint4(0, 0, 0, 0);
          }
          zeroed = true;
        }
        if (zeroed) fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars.kv_full[b], (uint32_t)nvalid * 4u * 2048u);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (blk[j] < 0) continue;
          tma_load_4d(st + 0 * kHalf + j * 2048, &kmap, &bars.kv_full[b], 0, h, 0, blk[j]);
          tma_load_4d(st + 1 * kHalf + j * 2048, &kmap, &bars.kv_full[b], 64, h, 0, blk[j]);
          tma_load_4d(st + 2 * kHalf + j * 2048, &vmap, &bars.kv_full[b], 0, h, 0, blk[j]);
          tma_load_4d(st + 3 * kHalf + j * 2048, &vmap, &bars.kv_full[b], 64, h, 0, blk[j]);
        }
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      if (!mbar_wait(&bars.q_full, 0)) timed_out = true;
      const uint32_t qa = smem_u32(smem + OFF_Q);
      const uint32_t pa_ = smem_u32(smem + OFF_P);
      for (int kt = 0; kt <= nkt && !timed_out; ++kt) {
        if (kt < nkt) {
          const int b = kt & 1;
          if (!mbar_wait(&bars.kv_full[b], (kt >> 1) & 1) ||
              (kt >= 2 && !mbar_wait(&bars.s_free[b], ((kt - 2) >> 1) & 1))) {
            timed_out = true;
            break;
          }
          tc::fence_after_sync();
          const uint32_t ka = smem_u32(smem + OFF_KV + b * STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            tc::mma_f16(tmem + b * 128, tc::desc_sw128(qa + off, 16, 1024), tc::desc_sw128(ka + off, 16, 1024),
                        IDESC_S, kk > 0);
          }
          tc::commit(&bars.s_full[b]);
        }
        if (kt >= 1) {
          const int j = kt - 1, b = j & 1;
          if (!mbar_wait(&bars.p_full, j & 1)) {
            timed_out = true;
            break;
          }
          tc::fence_after_sync();
          const uint32_t va = smem_u32(smem + OFF_KV + b * STAGE_BYTES + 2 * kHalf);
#pragma unroll
          for (int kk = 0; kk < 16; ++kk) {  // P_hi (kk < 8), then P_lo, against the same V
            const uint32_t aoff = (kk >> 3) * 2 * kHalf + ((kk >> 2) & 1) * kHalf + (kk & 3) * 32;
            tc::mma_f16(tmem + 256 + b * 128, tc::desc_sw128(pa_ + aoff, 16, 1024),
                        tc::desc_sw128(va + (kk & 7) * 2048, kHalf, 1024), IDESC_O, kk > 0);
          }
          tc::commit(&bars.pv_done[b]);
        }
      }
    }
  } else {
    // ---------------- softmax + epilogue (warps 0..3) ----------------
    const int r = threadIdx.x;
    const int tq = t0 + r / G;                       // query token within the chunk
    const int head = h * G + r % G;
    const int lim = min(start + tq, ctx - 1);        // last visible key position of this row
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f, alpha = 0.f;
    float o[128];
#pragma unroll
    for (int j = 0; j < 128; ++j) o[j] = 0.f;
    uint8_t *prow = smem + OFF_P + r * 128;

    for (int kt = 0; kt < nkt; ++kt) {
      const int b = kt & 1;
      if (!mbar_wait(&bars.s_full[b], (kt >> 1) & 1)) {
        timed_out = true;
        break;
      }
      tc::fence_after_sync();
      const uint32_t s_addr = tmem + lane_base + b * 128;
      const int kbase = kt * 128;

      float mx = -INFINITY;
#pragma unroll
      for (int cch = 0; cch < 4; ++cch) {
        uint32_t v[32];
        tc::ld_32x32b_x32(s_addr + cch * 32, v);
        tc::wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (kbase + cch * 32 + j <= lim) mx = fmaxf(mx, __uint_as_float(v[j]));
      }
      const float m_new = fmaxf(m_run, mx * sl2);
      const float a_new = exp2f(m_run - m_new);

      if (kt >= 1) {  // fold the previous tile's P V in before P is overwritten
        const int j = kt - 1;
        if (!mbar_wait(&bars.pv_done[j & 1], (j >> 1) & 1)) {
          timed_out = true;
          break;
        }
        tc::fence_after_sync();
        accumulate_o(o, tmem + lane_base + 256 + (j & 1) * 128, alpha);
      }

      float ls = 0.f;
#pragma unroll
      for (int cch = 0; cch < 4; ++cch) {
        uint32_t v[32];
        tc::ld_32x32b_x32(s_addr + cch * 32, v);
        tc::wait_ld();
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          const int key = kbase + cch * 32 + j;
          const float p0 = (key <= lim) ? exp2f(fmaf(__uint_as_float(v[j]), sl2, -m_new)) : 0.f;
          const float p1 = (key + 1 <= lim) ? exp2f(fmaf(__uint_as_float(v[j + 1]), sl2, -m_new)) : 0.f;
          ls += p0 + p1;
          hi[j >> 1] = Pack<T>::from_f2(p0, p1);
          const float2 h2 = Pack<T>::to_f2(hi[j >> 1]);
          lo[j >> 1] = Pack<T>::from_f2(p0 - h2.x, p1 - h2.y);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int q = cch * 4 + i, half = q >> 3, cc = q & 7;
          uint8_t *dst = prow + half * kHalf + ((cc ^ (r & 7)) << 4);
          *reinterpret_cast<uint4 *>(dst) = make_uint4(hi[4 * i], hi[4 * i + 1], hi[4 * i + 2], hi[4 * i + 3]);
          *reinterpret_cast<uint4 *>(dst + 2 * kHalf) =
              make_uint4(lo[4 * i], lo[4 * i + 1], lo[4 * i + 2], lo[4 * i + 3]);
        }
      }
      l_run = l_run * a_new + ls;
      m_run = m_new;
      alpha = a_new;
      tc::fence_before_sync();
      mbar_arrive(&bars.s_free[b]);

      if (kt == kt_ctx) {
        // value rows of keys >= ctx (partial last page, pages past the end)
        if (!mbar_wait(&bars.kv_full[b], (kt >> 1) & 1)) {
          timed_out = true;
          break;
        }
        const int z0 = ctx - kbase;
        uint8_t *vbase = smem + OFF_KV + b * STAGE_BYTES + 2 * kHalf;
        for (int idx = r; idx < (128 - z0) * 16; idx += 128) {
          const int row = z0 + (idx >> 4), part = idx & 15;
          *reinterpret_cast<uint4 *>(vbase + (part >> 3) * kHalf + row * 128 + (part & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars.p_full);
    }

    if (!timed_out) {
      const int j = nkt - 1;
      if (mbar_wait(&bars.pv_done[j & 1], (j >> 1) & 1)) {
        tc::fence_after_sync();
        accumulate_o(o, tmem + lane_base + 256 + (j & 1) * 128, alpha);
        if (tq < len) {
          const float inv = 1.f / l_run;
          T *op = reinterpret_cast<T *>(p.out) + ((int64_t)(row0 + tq) * p.num_q_heads + head) * kHeadDim;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            uint4 v;
            v.x = Pack<T>::from_f2(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
            v.y = Pack<T>::from_f2(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
            v.z = Pack<T>::from_f2(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
            v.w = Pack<T>::from_f2(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
            *reinterpret_cast<uint4 *>(op + 8 * i) = v;
          }
        }
      } else {
        timed_out = true;
      }
    }
  }

  if (timed_out) set_error(p.err, PA_ERR_TIMEOUT, c);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 5) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  griddep_launch_dependents();
}

template <typename T, int G>
cudaError_t launch_typed(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                         const CUtensorMap &qmap, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SMEM_BYTES);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  constexpr int TQ = 128 / G;
  dim3 grid((p.max_chunk_len + TQ - 1) / TQ, p.num_kv_heads, p.num_chunks);
  return launch_pdl(prefill_kernel<T, G>, grid, dim3(kThreads), SMEM_BYTES, stream, kmap, vmap, qmap, p);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                           const CUtensorMap &qmap, int dtype, int group, cudaStream_t stream) {
#define PA_PREFILL_CASE(T, G) \
  if (group == G) return launch_typed<T, G>(p, kmap, vmap, qmap, stream);
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
