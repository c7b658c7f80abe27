// Causal chunked prefill over an 8-bit KV pool (int8 codes or E4M3 codes,
// one fp32 scale per token and KV head; page "Модуль 04: KV-кэш и арифметика
// памяти", section 5, KV8Cache, and section 5.4), on mma.sync tensor cores.
//
// Computes what the 16-bit prefill computes (page "Модуль 12: Финальный
// проект: мини-движок инференса", qwen_serve/model.py, Qwen3Model.forward
// with T > 1: query token i of chunk c, at absolute position P + i, attends
// to keys 0 .. P + i of its KV head through the chunk's block table), with
// every key and value the dequantised number code * scale.
//
// One CTA takes one tile of 128 query rows for one KV head (128 / G tokens x
// the G query heads of that KV head, row r = token t0 + r / G, head
// h G + r % G), as the 16-bit prefill does, so every page read serves all G
// heads.  Eight compute warps own 16 rows each; a ninth warp streams the
// tile's pages (16 keys: K codes, V codes and both scale rows, 4224 bytes)
// through a ring of shared-memory stages with TMA, each stage released when
// all eight warps are done with it.  Per page a compute warp runs, with
// mma.sync m16n8k16 (fp16 operands, fp32 accumulators):
//   S = Q K^T   16 rows x 16 keys over the 128 dims (lane (g, t) = (lane / 4,
//               lane % 4) takes dims 32 t + 4 ks .. + 3 at k-step ks, so its
//               K operand is 32 contiguous code bytes of key g of the n-tile);
//               Q is the 16-bit input times a power of two per row (exact in
//               fp16), codes are exact in fp16 (E4M3 by the hardware
//               conversion, int8 as c + 1152 with the offset taken out of the
//               score: 1152 times the row's sum), every product is exact;
//   softmax     the score times the row's and the key's scales, masked past
//               the row's position; online per row (maximum and sum over the
//               four lanes that hold a row), the accumulators rescaled when a
//               row's maximum moves;
//   O += P V    P stays in registers (S's accumulator fragment is the A
//               fragment of this product), each weight times its value's
//               scale over a power-of-two unit R (raised, with the
//               accumulators, whenever a page's largest value scale passes
//               R 2^12); int8 values enter as c + 1152, whose offset (1152
//               times the sum of the fp16 weights) the epilogue subtracts.
// The epilogue divides by the row sum, multiplies by R and stores the rows
// of the chunk (lane t of a row holds its dims 32 t .. 32 t + 31).
#include <type_traits>

#include "pa_device.cuh"

namespace pa {
namespace {

constexpr int kWarps8 = 8;                      // compute warps, 16 rows each
constexpr int kThreads8 = (kWarps8 + 1) * 32;   // + the page producer
constexpr int kStages8 = 24;                    // page stages
// A stage: K codes (16 keys x 128) at 0, V codes at 2048, the 16 K scales at
// 4096, the 16 V scales at 4160 (the 8-bit decode's page layout).
constexpr int kPgV = 2048, kPgKS = 4096, kPgVS = 4160, kPgBytes = 4224;
constexpr int kStageStride8 = (kPgBytes + 127) / 128 * 128;
constexpr int OFF8_BAR = kStages8 * kStageStride8;
constexpr int SMEM8 = OFF8_BAR + kStages8 * (8 + 8 + 4) + 1024;
constexpr float kBias8 = 1152.f;                // int8 code c as the fp16 number c + 1152
constexpr unsigned FULL8 = 0xffffffffu;

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// Codes 0, 1 (I = 0) or 2, 3 (I = 1) of the word w as an fp16 pair: E4M3
// numbers exactly (hardware conversion of one 16-bit half), int8 codes c as
// c + 1152 (the byte c + 128 under the exponent of 1024).
template <bool F8, int I>
__device__ __forceinline__ uint32_t pair_h2(uint32_t w) {
  if constexpr (F8) {
    uint32_t r;
    if constexpr (I == 0)
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(w));
    else
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, hi;\n\t}" : "=r"(r) : "r"(w));
    return r;
  } else {
    return __byte_perm(w ^ 0x80808080u, 0x64646464u, I ? 0x4342u : 0x4140u);
  }
}

__device__ __forceinline__ uint32_t h2_pack(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&h);
}
__device__ __forceinline__ float2 h2_unpack(uint32_t u) {
  return __half22float2(*reinterpret_cast<const __half2 *>(&u));
}

template <typename T, int G, bool F8>
__global__ void __launch_bounds__(kThreads8, 1)
prefill8_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                const PrefillParams p) {
  constexpr int TQ = 128 / G;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + OFF8_BAR);
  uint64_t *empty = full + kStages8;
  int32_t *bad = reinterpret_cast<int32_t *>(empty + kStages8);  // per stage: its page was not loaded
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // heaviest tiles first: last chunk, last query tile
  const int c = p.num_chunks - 1 - (int)blockIdx.z;
  const int h = blockIdx.y;
  const int mt = (int)gridDim.x - 1 - (int)blockIdx.x;
  const int start = __ldg(p.chunk_starts + c), len = __ldg(p.chunk_lens + c), ctx = __ldg(p.context_lens + c);
  int row0 = 0;
  for (int i = 0; i < c; ++i) row0 += __ldg(p.chunk_lens + i);
  if (len < 1 || len > p.max_chunk_len || start < 0 || ctx != start + len || ctx > p.max_blocks_per_seq * kBlock ||
      row0 + len > p.total_q_tokens) {
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
  const int npg = last_key / kBlock + 1;                   // pages 0 .. npg - 1

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    for (int i = 0; i < kStages8; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kWarps8);
    }
    fence_mbar_init();
  }
  __syncthreads();
  bool timed_out = false;

  if (warp == kWarps8) {
    // ---------------- producer: pages 0 .. npg - 1 through the ring ----------------
    griddep_wait();  // the pool may come from the previous kernel (the 8-bit write)
    const int32_t *bt = p.block_tables + (int64_t)c * p.max_blocks_per_seq;
    int32_t win = -1;
    int issued = 0;
    for (int i = 0; i < npg; ++i) {
      const int st = i % kStages8;
      if (i >= kStages8 && !mbar_wait(&empty[st], ((i / kStages8) - 1) & 1)) {
        timed_out = true;
        break;
      }
      if ((i & 31) == 0) win = (i + lane < npg) ? __ldg(bt + i + lane) : -1;
      const int blk = __shfl_sync(FULL8, win, i & 31);
      const bool ok = (unsigned)blk < (unsigned)p.num_blocks;
      if (lane == 0) {
        uint8_t *dst = smem + st * kStageStride8;
        bad[st] = ok ? 0 : 1;
        if (ok) {
          mbar_arrive_expect_tx(&full[st], kPgBytes);
          tma_load_4d(dst, &kmap, &full[st], 0, h, 0, blk);
          tma_load_4d(dst + kPgV, &vmap, &full[st], 0, h, 0, blk);
          const int64_t si = ((int64_t)blk * p.num_kv_heads + h) * kBlock;  // the page's 16 scales: 64 bytes
          bulk_load(dst + kPgKS, p.k_scale + si, kBlock * 4, &full[st]);
          bulk_load(dst + kPgVS, p.v_scale + si, kBlock * 4, &full[st]);
        } else {
          set_error(p.err, PA_ERR_RANGE, c);
          mbar_arrive(&full[st]);  // (the arrival publishes bad[st]) the page is skipped
        }
      }
      issued = i + 1;
    }
    if (timed_out)  // a short, bounded chance for the copies in flight to land
      for (int i = issued - kStages8 > 0 ? issued - kStages8 : 0; i < issued; ++i)
        mbar_wait(&full[i % kStages8], (i / kStages8) & 1, kWaitLimitNs / 8);
  } else {
    // ---------------- compute warp: rows 16 warp + g and + 8 ----------------
    const int g = lane >> 2, t = lane & 3;
    int tq[2], pos[2];
    const T *qrow[2];
    for (int j = 0; j < 2; ++j) {
      const int r = 16 * warp + g + 8 * j;
      tq[j] = t0 + r / G;
      pos[j] = start + tq[j];  // the row's absolute position: it sees keys 0 .. pos
      qrow[j] = reinterpret_cast<const T *>(p.q) + ((int64_t)(row0 + tq[j]) * p.num_q_heads + h * G + r % G) * kHeadDim;
    }
    griddep_wait();  // q may come from the previous kernel
    // Q as the A operand: k-step ks holds dims 32 t + 4 ks + {0, 1} (regs 0, 1: rows g, g + 8) and
    // + {2, 3} (regs 2, 3); each row times 2^e so that its largest magnitude lies in [2^14, 2^15)
    uint32_t qa[8][4];
    float qsc[2], qbias[2];
    for (int j = 0; j < 2; ++j) {
      float f[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) f[i] = 0.f;
      if (tq[j] < len) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 u = *reinterpret_cast<const uint4 *>(qrow[j] + t * 32 + i * 8);
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
      amax = fmaxf(amax, __shfl_xor_sync(FULL8, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(FULL8, amax, 2));
      int e = amax > 0.f ? 141 - (int)((__float_as_uint(amax) >> 23) & 0xff) : 0;
      e = max(-120, min(120, e));
      const float sc = __uint_as_float((uint32_t)(127 + e) << 23);
      qsc[j] = p.scale_log2 * __uint_as_float((uint32_t)(127 - e) << 23);
      float qs = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa[ks][j] = h2_pack(f[4 * ks] * sc, f[4 * ks + 1] * sc);
        qa[ks][2 + j] = h2_pack(f[4 * ks + 2] * sc, f[4 * ks + 3] * sc);
        const float2 x = h2_unpack(qa[ks][j]), y = h2_unpack(qa[ks][2 + j]);
        qs += (x.x + x.y) + (y.x + y.y);
      }
      qs += __shfl_xor_sync(FULL8, qs, 1);
      qs += __shfl_xor_sync(FULL8, qs, 2);
      qbias[j] = F8 ? 0.f : kBias8 * qs;
    }

    float acc[16][4];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f}, ps[2] = {0.f, 0.f};
    float R = 0.f;
    // keys this warp's rows all see, and beyond which none sees
    const int pos_lo = start + t0 + (16 * warp) / G, pos_hi = start + t0 + (16 * warp + 15) / G;

    for (int i = 0; i < npg && !timed_out; ++i) {
      const int st = i % kStages8;
      if (!mbar_wait(&full[st], (i / kStages8) & 1)) {
        timed_out = true;
        break;
      }
      const uint8_t *kst = smem + st * kStageStride8;
      const int kb = i * kBlock;  // the page's first key position
      if (!bad[st] && kb <= pos_hi) {
        const uint8_t *vst = kst + kPgV;
        const float *kscale = reinterpret_cast<const float *>(kst + kPgKS);
        const float *vscale = reinterpret_cast<const float *>(kst + kPgVS);
        // ---- S: rows g, g + 8 x keys 2t, 2t + 1 (n-tile 0), 2t + 8, 2t + 9 (n-tile 1) ----
        uint32_t kw[2][8];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const uint4 *krow = reinterpret_cast<const uint4 *>(kst + (nt * 8 + g) * kHeadDim + t * 32);
          const uint4 k0 = krow[0], k1 = krow[1];
          kw[nt][0] = k0.x; kw[nt][1] = k0.y; kw[nt][2] = k0.z; kw[nt][3] = k0.w;
          kw[nt][4] = k1.x; kw[nt][5] = k1.y; kw[nt][6] = k1.z; kw[nt][7] = k1.w;
        }
        float cs[2][2][4] = {};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t b[2] = {pair_h2<F8, 0>(kw[nt][ks]), pair_h2<F8, 1>(kw[nt][ks])};
            mma16816(cs[nt][ks & 1], qa[ks], b);
          }
        }
        const float2 ks01 = *reinterpret_cast<const float2 *>(kscale + 2 * t);
        const float2 ks23 = *reinterpret_cast<const float2 *>(kscale + 8 + 2 * t);
        const float ksc[4] = {ks01.x, ks01.y, ks23.x, ks23.y};
        const bool whole = kb + kBlock - 1 <= pos_lo;  // (warp-uniform) every row sees every key of the page
        float s[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int nt = k >> 1, col = k & 1;
            const float v = cs[nt][0][2 * j + col] + cs[nt][1][2 * j + col] - qbias[j];
            const int key = kb + nt * 8 + 2 * t + col;
            s[j][k] = (whole || key <= pos[j]) ? v * (qsc[j] * ksc[k]) : -INFINITY;
          }
        // ---- online softmax per row (the quad of lanes 4 g .. 4 g + 3 holds a row's 16 keys) ----
        float alpha[2], pr[2][4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float mx = fmaxf(fmaxf(s[j][0], s[j][1]), fmaxf(s[j][2], s[j][3]));
          mx = fmaxf(mx, __shfl_xor_sync(FULL8, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(FULL8, mx, 2));
          const float mn = fmaxf(m[j], mx);
          const float base = mn == -INFINITY ? 0.f : mn;  // no visible key yet: every P is 0
          alpha[j] = ex2(m[j] - base);                      // 0 while nothing was accumulated
#pragma unroll
          for (int k = 0; k < 4; ++k) pr[j][k] = ex2(s[j][k] - base);
          l[j] = l[j] * alpha[j] + ((pr[j][0] + pr[j][1]) + (pr[j][2] + pr[j][3]));
          m[j] = mn;
        }
        // ---- value scales against the unit R ----
        const float2 vs01 = *reinterpret_cast<const float2 *>(vscale + 2 * t);
        const float2 vs23 = *reinterpret_cast<const float2 *>(vscale + 8 + 2 * t);
        float vmax = fmaxf(fmaxf(vs01.x, vs01.y), fmaxf(vs23.x, vs23.y));
        vmax = fmaxf(vmax, __shfl_xor_sync(FULL8, vmax, 1));
        vmax = fmaxf(vmax, __shfl_xor_sync(FULL8, vmax, 2));  // all 16 keys, the same in every lane
        float rs = 1.f;
        if (vmax > R * 4096.f) {
          const float Rn = __uint_as_float((__float_as_uint(vmax) + 0x007fffffu) & 0xff800000u);
          rs = R / Rn;
          R = Rn;
        }
        const float invR = __uint_as_float((254u << 23) - __float_as_uint(R));
        const float f0 = alpha[0] * rs, f1 = alpha[1] * rs;
        if (__any_sync(FULL8, f0 != 1.f || f1 != 1.f)) {
#pragma unroll
          for (int nt = 0; nt < 16; ++nt) {
            acc[nt][0] *= f0;
            acc[nt][1] *= f0;
            acc[nt][2] *= f1;
            acc[nt][3] *= f1;
          }
        }
        const float vsc[4] = {vs01.x * invR, vs01.y * invR, vs23.x * invR, vs23.y * invR};
        // P'' as the A operand: rows g (regs 0, 2), g + 8 (regs 1, 3); keys 2t, 2t + 1 then 2t + 8, 2t + 9
        uint32_t pa[4];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          pa[j] = h2_pack(pr[j][0] * vsc[0], pr[j][1] * vsc[1]);
          pa[2 + j] = h2_pack(pr[j][2] * vsc[2], pr[j][3] * vsc[3]);
          if constexpr (!F8) {  // the weights as the product sees them, for the int8 offset
            const float2 x = h2_unpack(pa[j]), y = h2_unpack(pa[2 + j]);
            ps[j] = ps[j] * (alpha[j] * rs) + ((x.x + x.y) + (y.x + y.y));
          }
        }
        // ---- O += P V: value rows of keys 2t, 2t + 1, 2t + 8, 2t + 9 at dims 16 g .. 16 g + 15 ----
        uint4 v0 = *reinterpret_cast<const uint4 *>(vst + (2 * t) * kHeadDim + 16 * g);
        uint4 v1 = *reinterpret_cast<const uint4 *>(vst + (2 * t + 1) * kHeadDim + 16 * g);
        uint4 v2 = *reinterpret_cast<const uint4 *>(vst + (2 * t + 8) * kHeadDim + 16 * g);
        uint4 v3 = *reinterpret_cast<const uint4 *>(vst + (2 * t + 9) * kHeadDim + 16 * g);
        if (kb + kBlock > ctx) {  // slots past the sequence may hold any bytes (an E4M3 NaN): zero them
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          if (kb + 2 * t >= ctx) v0 = z;
          if (kb + 2 * t + 1 >= ctx) v1 = z;
          if (kb + 2 * t + 8 >= ctx) v2 = z;
          if (kb + 2 * t + 9 >= ctx) v3 = z;
        }
        const uint32_t w0[4] = {v0.x, v0.y, v0.z, v0.w}, w1[4] = {v1.x, v1.y, v1.z, v1.w};
        const uint32_t w2[4] = {v2.x, v2.y, v2.z, v2.w}, w3[4] = {v3.x, v3.y, v3.z, v3.w};
#pragma unroll
        for (int np = 0; np < 8; ++np) {  // n-tiles 2 np, 2 np + 1: dims 16 g + 2 np, + 1 of each column group
          const uint32_t sel = (np & 1) ? 0x7362u : 0x5140u;
          const uint32_t x = __byte_perm(w0[np >> 1], w1[np >> 1], sel);
          const uint32_t y = __byte_perm(w2[np >> 1], w3[np >> 1], sel);
          const uint32_t b0[2] = {pair_h2<F8, 0>(x), pair_h2<F8, 0>(y)};
          const uint32_t b1[2] = {pair_h2<F8, 1>(x), pair_h2<F8, 1>(y)};
          mma16816(acc[2 * np], pa, b0);
          mma16816(acc[2 * np + 1], pa, b1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---- epilogue: rows of the chunk; lane t holds dims 32 t + nt (acc[nt][2j]) and 32 t + 16 + nt ----
    if (!timed_out) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float lt = l[j], pt = ps[j];
        lt += __shfl_xor_sync(FULL8, lt, 1);
        lt += __shfl_xor_sync(FULL8, lt, 2);
        pt += __shfl_xor_sync(FULL8, pt, 1);
        pt += __shfl_xor_sync(FULL8, pt, 2);
        if (tq[j] < len) {
          const float f = R / lt, off = kBias8 * pt;
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float a0 = acc[2 * i][2 * j], a1 = acc[2 * i + 1][2 * j];
            float b0 = acc[2 * i][2 * j + 1], b1 = acc[2 * i + 1][2 * j + 1];
            if constexpr (!F8) {
              a0 -= off; a1 -= off; b0 -= off; b1 -= off;
            }
            pk[i] = Pack<T>::from_f2(a0 * f, a1 * f);      // dims 32 t + 2 i, + 1
            pk[8 + i] = Pack<T>::from_f2(b0 * f, b1 * f);  // dims 32 t + 16 + 2 i, + 1
          }
          T *op = reinterpret_cast<T *>(p.out) +
                  ((int64_t)(row0 + tq[j]) * p.num_q_heads + h * G + (16 * warp + g + 8 * j) % G) * kHeadDim + 32 * t;
          uint4 *o4 = reinterpret_cast<uint4 *>(op);
          o4[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          o4[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          o4[2] = make_uint4(pk[8], pk[9], pk[10], pk[11]);
          o4[3] = make_uint4(pk[12], pk[13], pk[14], pk[15]);
        }
      }
    }
  }
  if (timed_out) set_error(p.err, PA_ERR_TIMEOUT, c);
  __syncthreads();  // no stage is read or written once the CTA ends
  griddep_launch_dependents();
}

template <typename T, int G, bool F8>
cudaError_t launch8(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap, cudaStream_t stream) {
  static KernelSetup setup;
  cudaError_t e = kernel_setup(setup, prefill8_kernel<T, G, F8>, SMEM8, kThreads8, nullptr);
  if (e != cudaSuccess) return e;
  constexpr int TQ = 128 / G;
  dim3 grid((p.max_chunk_len + TQ - 1) / TQ, p.num_kv_heads, p.num_chunks);
  return launch_pdl(prefill8_kernel<T, G, F8>, grid, dim3(kThreads8), SMEM8, stream, kmap, vmap, p);
}

}  // namespace

cudaError_t launch_prefill8(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap, int dtype,
                            int group, bool f8, cudaStream_t stream) {
#define PA_P8_CASE(T, G)                                                  \
  if (group == G) return f8 ? launch8<T, G, true>(p, kmap, vmap, stream) \
                            : launch8<T, G, false>(p, kmap, vmap, stream);
  if (dtype == PA_BF16) {
    PA_P8_CASE(__nv_bfloat16, 1)
    PA_P8_CASE(__nv_bfloat16, 2)
    PA_P8_CASE(__nv_bfloat16, 4)
    PA_P8_CASE(__nv_bfloat16, 8)
  } else {
    PA_P8_CASE(__half, 1)
    PA_P8_CASE(__half, 2)
    PA_P8_CASE(__half, 4)
    PA_P8_CASE(__half, 8)
  }
#undef PA_P8_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
