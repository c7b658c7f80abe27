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
// Keys stream in tiles of N = 128 (8 pages, one TMA box per page and 64-dim
// half), double-buffered.  Per key tile kt:
//   S = Q K^T     tcgen05.mma kind::f16, A and B from shared memory (K-major),
//                 fp32 into TMEM columns S[kt % 2].
//   softmax       8 warps: the two warps on TMEM lane quarter q own rows
//                 32q .. 32q + 31, one the keys 0..63 and the other 64..127
//                 of the tile; they exchange row maxima through shared memory.
//                 P = exp2(S * scale * log2 e - m) is written back into the
//                 same TMEM columns as two terms of the input dtype, P_hi =
//                 round(P) and P_lo = round(P - P_hi) (each 32-key chunk of S
//                 becomes 16 columns of P_hi pairs then 16 of P_lo pairs, so
//                 no S value is overwritten before it is read).
//   O += P V      tcgen05.mma with A = P_hi, then P_lo, read from TMEM, and B =
//                 the V tile (MN-major) from shared memory; O (fp32) stays in
//                 TMEM for the whole key loop.
// m is a per-row reference maximum: it only moves (rescaling O in TMEM and the
// row sum) when a tile's maximum exceeds it by more than 2^8, so O is rarely
// touched by the threads.  Warp 8 issues the TMA loads, warp 9 owns TMEM and
// issues the MMAs (one thread each); mbarriers hand tiles between the roles
// and every wait is bounded.  Keys above the diagonal are masked per element
// on the tiles that cross it (a warp-uniform test picks the unmasked path
// elsewhere) and never loaded past the tile holding the tile's last query.
// Value rows past the sequence's last key are zeroed in shared memory before
// the PV product so that a zero probability never meets a non-finite value.
#include <type_traits>

#include "tcgen05.cuh"

namespace pa {
namespace {

constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kWarpTma = kSoftmaxWarps, kWarpMma = kSoftmaxWarps + 1;
constexpr int kThreads = (kSoftmaxWarps + 2) * 32;
constexpr int kHalf = 16384;                       // 128 rows x 64 elements x 2 bytes
constexpr int kStages = 2;
constexpr int OFF_Q = 0;                           // Q: two 64-dim halves
constexpr int OFF_KV = 2 * kHalf;                  // stages of {K lo, K hi, V lo, V hi}
constexpr int STAGE_BYTES = 4 * kHalf;
constexpr int OFF_X = OFF_KV + kStages * STAGE_BYTES;  // row-max / row-sum exchange [2][2][128] fp32
constexpr int OFF_BAR = OFF_X + 2 * 2 * 128 * 4;
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;   // + barriers (< 256 B) + alignment slack   // + barriers + alignment slack
constexpr uint32_t kTmemCols = 512;                // S/P 0, S/P 1, O, (unused)
constexpr uint32_t kColO = 256;
constexpr float kRescale = 8.f;                    // log2 of the largest P before O is rescaled

// Every barrier that signals once per key tile comes in a pair indexed by the
// tile's parity, so no waiter can be overtaken by two phases.
struct Bars {
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t x_full[2];  // row-max / row-sum exchange between the two halves of a row
  uint32_t tmem_base;
};

template <typename T, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap qmap, const PrefillParams p) {
  constexpr int TQ = 128 / G;  // query tokens per tile
  constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t IDESC_S = tc::idesc_f16(kBF16, 128, 128, false);
  constexpr uint32_t IDESC_O = tc::idesc_f16(kBF16, 128, 128, true);
  constexpr unsigned FULL = 0xffffffffu;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars &bars = *reinterpret_cast<Bars *>(smem + OFF_BAR);
  float *xbuf = reinterpret_cast<float *>(smem + OFF_X);
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
    for (int b = 0; b < kStages; ++b) mbar_init(&bars.kv_full[b], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.s_full[b], 1);
      mbar_init(&bars.pv_done[b], 1);
      mbar_init(&bars.p_full[b], kSoftmaxThreads);
      mbar_init(&bars.x_full[b], kSoftmaxThreads);
    }
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tc::tmem_alloc(&bars.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars.tmem_base;
  bool timed_out = false;

  if (warp == kWarpTma) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      mbar_arrive_expect_tx(&bars.q_full, 2 * kHalf);
      tma_load_3d(smem + OFF_Q, &qmap, &bars.q_full, 0, h * G, row0 + t0);
      tma_load_3d(smem + OFF_Q + kHalf, &qmap, &bars.q_full, 64, h * G, row0 + t0);
      for (int kt = 0; kt < nkt; ++kt) {
        const int b = kt % kStages;
        // the stage is free once the PV product of the tile that used it is done
        if (kt >= kStages) {
          const int j = kt - kStages;
          if (!mbar_wait(&bars.pv_done[j & 1], (j >> 1) & 1)) {
            timed_out = true;
            break;
          }
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
  } else if (warp == kWarpMma) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      if (!mbar_wait(&bars.q_full, 0)) timed_out = true;
      const uint32_t qa = smem_u32(smem + OFF_Q);
      for (int kt = 0; kt <= nkt && !timed_out; ++kt) {
        if (kt < nkt) {
          const int b = kt % kStages, sb = kt & 1;
          if (!mbar_wait(&bars.kv_full[b], (kt / kStages) & 1)) {
            timed_out = true;
            break;
          }
          tc::fence_after_sync();
          const uint32_t ka = smem_u32(smem + OFF_KV + b * STAGE_BYTES);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
            tc::mma_f16(tmem + sb * 128, tc::desc_sw128(qa + off, 16, 1024), tc::desc_sw128(ka + off, 16, 1024),
                        IDESC_S, kk > 0);
          }
          tc::commit(&bars.s_full[sb]);
        }
        if (kt >= 1) {  // O += P V of the previous tile
          const int j = kt - 1, sj = j & 1;
          if (!mbar_wait(&bars.p_full[sj], (j >> 1) & 1)) {
            timed_out = true;
            break;
          }
          tc::fence_after_sync();
          const uint32_t va = smem_u32(smem + OFF_KV + (j % kStages) * STAGE_BYTES + 2 * kHalf);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t a_hi = tmem + sj * 128 + 32 * (kk >> 1) + 8 * (kk & 1);
            const uint64_t bdesc = tc::desc_sw128(va + kk * 2048, kHalf, 1024);
            tc::mma_f16_ts(tmem + kColO, a_hi, bdesc, IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
            tc::mma_f16_ts(tmem + kColO, a_hi + 16, bdesc, IDESC_O, 1u);
          }
          tc::commit(&bars.pv_done[sj]);
        }
      }
    }
  } else {
    // ---------------- softmax + epilogue (warps 0..7) ----------------
    const int quad = warp & 3, ch = warp >> 2;       // TMEM lane quarter, key half of the tile
    const int r = quad * 32 + lane;                  // tile row = TMEM lane
    const int tid = warp * 32 + lane;                // 0 .. 255
    const int tq = t0 + r / G;                       // query token within the chunk
    const int head = h * G + r % G;
    const int lim = min(start + tq, ctx - 1);        // last visible key position of this row
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;

    for (int kt = 0; kt < nkt; ++kt) {
      const int sb = kt & 1;
      if (!mbar_wait(&bars.s_full[sb], (kt >> 1) & 1)) {
        timed_out = true;
        break;
      }
      tc::fence_after_sync();
      const uint32_t s_addr = tmem + lane_base + sb * 128 + ch * 64;
      const int kbase = kt * 128 + ch * 64;          // first key of this thread's half
      uint32_t v[2][32];
      tc::ld_32x32b_x32(s_addr, v[0]);
      tc::ld_32x32b_x32(s_addr + 32, v[1]);
      tc::wait_ld();
      const bool full = __all_sync(FULL, kbase + 63 <= lim);

      float mx = -INFINITY;
      if (full) {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int j = 0; j < 32; ++j) mx = fmaxf(mx, __uint_as_float(v[cc][j]));
      } else {
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (kbase + cc * 32 + j <= lim) mx = fmaxf(mx, __uint_as_float(v[cc][j]));
      }
      float *xb = xbuf + (kt & 1) * 256;
      xb[ch * 128 + r] = mx;
      mbar_arrive(&bars.x_full[kt & 1]);
      if (!mbar_wait(&bars.x_full[kt & 1], (kt >> 1) & 1)) {
        timed_out = true;
        break;
      }
      mx = fmaxf(mx, xb[(1 - ch) * 128 + r]);
      const float mc = mx * sl2;
      if (kt == 0) {
        m_ref = mc;  // every row sees key 0, so the first tile's maximum is finite
      } else {
        const bool need = mc > m_ref + kRescale;
        if (__any_sync(FULL, need)) {  // warp-uniform: the TMEM accesses below are warp-wide
          const float f = need ? exp2f(m_ref - mc) : 1.f;
          if (need) {
            l *= f;
            m_ref = mc;
          }
          // every earlier P V has landed in O: scale this thread's half of its row
          const int j = kt - 1;
          if (!mbar_wait(&bars.pv_done[j & 1], (j >> 1) & 1)) {
            timed_out = true;
            break;
          }
          tc::fence_after_sync();
          const uint32_t o_addr = tmem + lane_base + kColO + ch * 64;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t ov[32];
            tc::ld_32x32b_x32(o_addr + cc * 32, ov);
            tc::wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * f);
            tc::st_32x32b_x32(o_addr + cc * 32, ov);
          }
        }
      }

      // P in two terms of the input dtype, written over this half's S columns
      float ls = 0.f;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float s0 = __uint_as_float(v[cc][2 * j]), s1 = __uint_as_float(v[cc][2 * j + 1]);
          float p0 = exp2f(fmaf(s0, sl2, -m_ref));
          float p1 = exp2f(fmaf(s1, sl2, -m_ref));
          if (!full) {
            const int key = kbase + cc * 32 + 2 * j;
            p0 = (key <= lim) ? p0 : 0.f;
            p1 = (key + 1 <= lim) ? p1 : 0.f;
          }
          ls += p0 + p1;
          pk[j] = Pack<T>::from_f2(p0, p1);
          const float2 h2 = Pack<T>::to_f2(pk[j]);
          pk[16 + j] = Pack<T>::from_f2(p0 - h2.x, p1 - h2.y);
        }
        tc::st_32x32b_x32(s_addr + cc * 32, pk);
      }
      tc::wait_st();
      l += ls;

      if (kt == kt_ctx) {
        // value rows of keys >= ctx (partial last page, pages past the end)
        if (!mbar_wait(&bars.kv_full[kt % kStages], (kt / kStages) & 1)) {
          timed_out = true;
          break;
        }
        const int z0 = ctx - kt * 128;
        uint8_t *vbase = smem + OFF_KV + (kt % kStages) * STAGE_BYTES + 2 * kHalf;
        for (int idx = tid; idx < (128 - z0) * 16; idx += kSoftmaxThreads) {
          const int row = z0 + (idx >> 4), part = idx & 15;
          *reinterpret_cast<uint4 *>(vbase + (part >> 3) * kHalf + row * 128 + (part & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc::fence_before_sync();
      mbar_arrive(&bars.p_full[kt & 1]);
    }

    if (!timed_out) {
      const int j = nkt - 1;
      if (mbar_wait(&bars.pv_done[j & 1], (j >> 1) & 1)) {
        tc::fence_after_sync();
        // row sum: the two halves exchange theirs (next phase of the exchange barriers)
        float *xl = xbuf + (nkt & 1) * 256;
        xl[ch * 128 + r] = l;
        mbar_arrive(&bars.x_full[nkt & 1]);
        if (mbar_wait(&bars.x_full[nkt & 1], (nkt >> 1) & 1)) {
          const float inv = 1.f / (l + xl[(1 - ch) * 128 + r]);
          T *op = reinterpret_cast<T *>(p.out) + ((int64_t)(row0 + tq) * p.num_q_heads + head) * kHeadDim + ch * 64;
          const uint32_t o_addr = tmem + lane_base + kColO + ch * 64;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t ov[32];
            tc::ld_32x32b_x32(o_addr + cc * 32, ov);  // warp-wide; only rows of the chunk are stored
            tc::wait_ld();
            if (tq < len) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint4 w;
                w.x = Pack<T>::from_f2(__uint_as_float(ov[8 * i + 0]) * inv, __uint_as_float(ov[8 * i + 1]) * inv);
                w.y = Pack<T>::from_f2(__uint_as_float(ov[8 * i + 2]) * inv, __uint_as_float(ov[8 * i + 3]) * inv);
                w.z = Pack<T>::from_f2(__uint_as_float(ov[8 * i + 4]) * inv, __uint_as_float(ov[8 * i + 5]) * inv);
                w.w = Pack<T>::from_f2(__uint_as_float(ov[8 * i + 6]) * inv, __uint_as_float(ov[8 * i + 7]) * inv);
                *reinterpret_cast<uint4 *>(op + cc * 32 + 8 * i) = w;
              }
            }
          }
        } else {
          timed_out = true;
        }
      } else {
        timed_out = true;
      }
    }
  }

  if (timed_out) set_error(p.err, PA_ERR_TIMEOUT, c);
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
