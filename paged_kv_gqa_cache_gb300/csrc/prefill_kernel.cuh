#pragma once
// Causal chunked-prefill attention over a paged KV cache on the tcgen05
// tensor cores (sm_103a).
//
// For chunk c (start P, n new tokens, context P + n), query token i at
// absolute position P + i and query head g attends to keys 0 .. P + i of KV
// head g / G, read through the chunk's block table (page "Модуль 12:
// Финальный проект: мини-движок инференса", qwen_serve/model.py,
// Qwen3Model.forward with T > 1: mask kpos <= qpos on absolute positions;
// page "Модуль 04: KV-кэш и арифметика памяти", section 3.4: the prefix KV
// lives in the cache between chunks).  With a sliding window of W keys
// (page "Модуль 04: KV-кэш и арифметика памяти", sections 4 and 5.2) the
// query at position p sees only keys p - W + 1 .. p: a tile's key loop starts
// at the key tile of its first row's lowest key, and pages wholly below that
// key are never read.
//
// One CTA computes one M = 128 tile of query rows for one KV head: 128 / G
// consecutive tokens of the chunk x the G query heads sharing that KV head,
// so every K/V tile it reads serves all G heads.  Row r of the tile is token
// t0 + r / G, head h * G + r % G (the Q tile is one TMA box per 64-dim half).
// Keys stream in tiles of N = 128 (8 pages; K as two 2 KB TMA boxes per page,
// the 64-dim halves of 16 keys, gathered half by half; V as one 4 KB box per
// page with its two halves 2 KB apart; 128-byte swizzled): K through a
// 3-stage ring released as soon as S is computed, V through a 3-stage ring
// released after the PV product.  Seven loader warps fill both rings, each
// issuing a seventh of every tile's 24 boxes from parallel lanes: the TMA engine
// serves each issuing warp at a fixed cost per box, so the box count and the
// warps, not the ring depth, set the ingest rate.  Per key tile kt:
//   S = Q K^T     tcgen05.mma kind::f16, A and B from shared memory (K-major),
//                 fp32 into TMEM columns S[kt % 2].
//   softmax       8 warps; the two warps on TMEM lane quarter q own rows
//                 32q .. 32q + 31, warp half 0 the keys 0..63 of every tile,
//                 half 1 the keys 64..127.  Each half keeps its own per-row
//                 reference maximum m, row sum l and output accumulator O_half,
//                 so the halves never synchronise inside the key loop.
//                 P = 2^(S * scale * log2 e - m) goes back into the same TMEM
//                 columns rounded to the input dtype, P_hi = round(P) (each
//                 32-key chunk of S becomes 16 columns of P_hi pairs, so no S
//                 value is overwritten before it is read).  Rows that see
//                 fewer than 128 keys (all of them in key tile 0) average the
//                 rounding errors of too few probabilities, so on key tile 0
//                 of a query tile that holds such rows P also gets its second
//                 term P_lo = round(P - P_hi), in the next 16 columns.
//   O_half += P V tcgen05.mma with A = P_hi (then P_lo where it exists), read
//                 from TMEM, and B = the V rows of that half (MN-major) from
//                 shared memory; both O accumulators (fp32) stay in TMEM for
//                 the whole key loop.
// m only moves (rescaling that half's O and l) when a tile's maximum exceeds
// it by more than 2^8, so the threads rarely touch O.  The epilogue merges the
// two halves of each row, O = O_0 2^(m_0 - M) + O_1 2^(m_1 - M) over
// l_0 2^(m_0 - M) + l_1 2^(m_1 - M), and stores it in the input dtype.
// Warps 8..14 load Q, K and V, warp 15 owns TMEM and issues the
// MMAs (one thread); mbarriers hand tiles between the roles and every wait is
// bounded.  Keys above the diagonal are masked per element on the tiles that
// cross it (a warp-uniform test picks the unmasked path elsewhere) and never
// loaded past the tile holding the tile's last query.  Value rows past the
// sequence's last key are zeroed in shared memory before the PV product so that
// a zero probability never meets a non-finite value.
//
// Over an 8-bit pool (CODES = 1: int8, 2: E4M3; page "Модуль 04: KV-кэш и
// арифметика памяти", section 5, KV8Cache, and section 5.4) the same kernel
// runs with f16 operands: the loader warps become converters (4 for K, 3 for
// V: S waits for K, while V has the softmax's time to spare), each fetching
// its pages' codes (one 2 KB TMA box per page, a tile ahead) into the stage
// and rewriting them in place as the f16 rows the MMAs read, code * scale
// rounded once to f16 (rows past the sequence become zeros); a bf16 query
// tile is rewritten as f16 after scaling each row by the power of two that
// puts its largest magnitude in [2^14, 2^15) (exact), the row's scale_log2
// taking the inverse power.  P is then f16 too; the output keeps the query
// dtype.
#include <type_traits>

#include "tcgen05.cuh"

namespace pa {
namespace {

constexpr int kSoftmaxWarps = 8;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kLoadWarps = 7;  // each issues a seventh of the 24 boxes of every K and V tile
constexpr int kWarpLoad0 = kSoftmaxWarps, kWarpMma = kSoftmaxWarps + kLoadWarps;
constexpr int kThreads = (kSoftmaxWarps + kLoadWarps + 1) * 32;
static_assert(kThreads == 512, "four warpgroups: two of softmax warps, two of loader and MMA warps");
// Registers: 128 per thread at launch (65536 / 512).  Inside their roles the
// softmax warpgroups take kRegsSoftmax and the loader / MMA warpgroups keep
// kRegsOther (2 x 128 x (kRegsSoftmax + kRegsOther) <= 65536, what the launch
// holds, so an increase never waits forever); every role gives its share back
// to 128 before the common tail.
constexpr int kRegsSoftmax = 200, kRegsOther = 56;
static_assert(2 * 128 * kRegsSoftmax + 2 * 128 * kRegsOther <= 65536, "register split fits the launch");
// Over 8-bit pools the converters hold two pages' codes and their conversions:
// 96 registers (the softmax keeping 160) is what they need without spilling.
constexpr int kRegsSoftmax8 = 160, kRegsOther8 = 96;
static_assert(2 * 128 * kRegsSoftmax8 + 2 * 128 * kRegsOther8 <= 65536, "register split fits the launch");
template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
// A warpgroup that gives registers up on entering its role and asks for them
// back at its end could, with little work, ask before the warpgroups that
// take those registers have taken them; their increase would then wait
// forever.  So the warpgroups that take registers arrive on a named barrier
// once they have them (regs_taken: no waiting), and the ones that gave them
// up wait on it before asking for them back (regs_wait_taken); every thread of
// the CTA passes the barrier exactly once.
constexpr int kRegsBarrier = 4;  // named barrier id (0: __syncthreads, 1-3: the roles' own)
__device__ __forceinline__ void regs_taken() {
  asm volatile("bar.arrive %0, %1;" ::"r"(kRegsBarrier), "r"(kThreads) : "memory");
}
__device__ __forceinline__ void regs_wait_taken() { named_barrier(kRegsBarrier, kThreads); }
constexpr int kHalf = 16384;                        // 128 rows x 64 elements x 2 bytes
constexpr int kVPage = 4096;                        // V: one page (16 rows x 128 dims x 2 bytes) per box
constexpr int kKStages = 3, kVStages = 3;
constexpr int OFF_Q = 0;                            // Q: two 64-dim halves
constexpr int OFF_K = 2 * kHalf;                    // K stages: {lo, hi} halves
constexpr int OFF_V = OFF_K + kKStages * 2 * kHalf; // V stages: {lo, hi} halves
constexpr int kBtCache = 256;                       // block ids of the chunk cached in shared memory
constexpr int OFF_BT = OFF_V + kVStages * 2 * kHalf;
constexpr int OFF_BAR = OFF_BT + kBtCache * 4;
// The epilogue runs once every QK^T product has completed, so it borrows the
// K ring: the (m, l) exchange [2][128] float2, then 1 KB of staging per softmax warp.
constexpr int OFF_X = OFF_K;
constexpr int OFF_STAGE = OFF_X + 2 * 128 * 8;
constexpr int kStageBytes = 1024;
static_assert(OFF_STAGE + kSoftmaxWarps * kStageBytes <= OFF_V, "epilogue areas fit in the K ring");
constexpr int SMEM_BYTES = OFF_BAR + 256 + 1024;    // + barriers (< 256 B) + alignment slack
static_assert(SMEM_BYTES <= 232448, "shared memory");
constexpr uint32_t kTmemCols = 512;                 // S/P 0, S/P 1, O_0, O_1
constexpr uint32_t kTmemAllocHere = 0xffffffffu;    // prefill_tile: allocate the columns in the tile's set-up
constexpr uint32_t kColO = 256;
constexpr float kRescale = 8.f;                     // log2 of the largest P before O is rescaled
constexpr float kRescaleSum = 256.f;                // 2^kRescale: a half-row sum at most this has no larger P

// Every per-tile barrier exists once per ring stage (tile kt uses stage
// kt % 3) and completes once per tile of that stage.  No waiter can be
// overtaken by two phases: the next tile of a stage needs, through the rings
// or the MMA order, the very step each waiter of the stage is waiting for.
static_assert(kKStages == kVStages, "QK^T and P V barriers share the stage index");
struct Bars {
  uint64_t q_full;
  uint64_t k_full[kKStages];   // K tile landed (one arrival per loader warp + TMA bytes)
  uint64_t v_full[kVStages];   // V tile landed
  uint64_t s_full[kKStages];   // QK^T of the tile done: S readable, K stage free
  uint64_t p_full[kVStages];   // P of the tile written by every softmax thread, each of which saw V land
  uint64_t pv_done[kVStages];  // P V of the tile done: O holds it, V stage free
  uint64_t x_full;
  uint64_t drain;              // timeout path only: every MMA issued so far has completed
  // 8-bit pools only
  uint64_t kc_full[kKStages];  // the K codes of the tile landed (one arrival per K converter + TMA bytes)
  uint64_t vc_full[kVStages];  // the V codes of the tile landed
  uint64_t q_conv;             // the query tile rewritten as f16 (bf16 queries)
  uint32_t tmem_base;
};
static_assert(sizeof(Bars) <= 256, "barriers");

// 8-bit pools: converter warps per operand, and one page of one KV head's codes
constexpr int kKConv = 4, kVConv = kLoadWarps - kKConv;
static_assert((8 + kKConv - 1) / kKConv <= 3 && (8 + kVConv - 1) / kVConv <= 3, "at most 3 pages per converter");
constexpr int kCodePage = 2048;  // 16 rows x 128 one-byte codes

// Key tile kt of the K pool is 16 boxes of 2 KB, box b being the 64-dim half
// b % 2 of page b / 2 (the QK^T product reads each half of all 128 keys as one
// K-major operand, so the halves of the 8 pages are gathered into two 16 KB
// blocks), fetched into `dst` and completing on `bar` (which expects one
// arrival per loader warp).  A TMA engine serves each issuing warp at about
// one small box per 50 ns, so the boxes are spread over the loader warps: this
// warp's lane i issues box b0 + kLoadWarps * i.  Pages past the sequence and
// pages below pg0 (wholly before the sliding window) are skipped: their keys
// are masked.  A page whose block id is out of range is zeroed and reported.
// sbt caches the block ids of pages pg0 ...
__device__ __forceinline__ void load_boxes(uint8_t *dst, const CUtensorMap *map, uint64_t *bar, int kt, int b0,
                                           int h, int pg0, int npages, const int32_t *sbt, const int32_t *bt,
                                           const PrefillParams &p, int c, int lane) {
  const int b = b0 + kLoadWarps * lane;
  const int page = b >> 1, half = b & 1;
  const int pg = kt * 8 + page;
  const bool in = b < 16 && pg >= pg0 && pg < npages;
  int id = -1;
  if (in) id = (sbt && pg - pg0 < kBtCache) ? sbt[pg - pg0] : __ldg(bt + pg);
  const bool ok = in && (unsigned)id < (unsigned)p.num_blocks;
  const unsigned okmask = __ballot_sync(0xffffffffu, ok);
  uint8_t *box = dst + half * kHalf + page * 2048;
  if (in && !ok) {  // rare: keep the products finite
    if (half == 0) set_error(p.err, PA_ERR_RANGE, c);  // the error word reports the chunk
    uint4 *z = reinterpret_cast<uint4 *>(box);
    for (int i = 0; i < 128; ++i) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  __syncwarp();  // the zeroed boxes are written before the arrival below releases them
  if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(okmask) * 2048u);
  __syncwarp();
  if (ok) tma_load_4d(box, map, bar, half * 64, h, 0, id);
}

// Key tile kt of the V pool is 8 boxes of 4 KB: page p (its 16 rows of dims
// 0..63, then of dims 64..127, 128-byte swizzled) at dst + 4 KB p, completing
// on `bar` (one arrival per loader warp).  This warp's lane i fetches page
// p0 + kLoadWarps * i.  Pages past the sequence are skipped (the softmax warps
// zero those rows); pages below pg0 (wholly before the sliding window) and
// pages whose block id is out of range (reported) are zeroed: their rows meet
// zero probabilities and must stay finite.
__device__ __forceinline__ void load_vpages(uint8_t *dst, const CUtensorMap *map, uint64_t *bar, int kt, int p0,
                                            int h, int pg0, int npages, const int32_t *sbt, const int32_t *bt,
                                            const PrefillParams &p, int c, int lane) {
  const int page = p0 + kLoadWarps * lane;
  const int pg = kt * 8 + page;
  const bool in = page < 8 && pg >= pg0 && pg < npages;
  int id = -1;
  if (in) id = (sbt && pg - pg0 < kBtCache) ? sbt[pg - pg0] : __ldg(bt + pg);
  const bool ok = in && (unsigned)id < (unsigned)p.num_blocks;
  const unsigned okmask = __ballot_sync(0xffffffffu, ok);
  uint8_t *box = dst + page * kVPage;
  if ((in && !ok) || (page < 8 && pg < pg0)) {  // rare
    if (in) set_error(p.err, PA_ERR_RANGE, c);  // the error word reports the chunk
    uint4 *z = reinterpret_cast<uint4 *>(box);
    for (int i = 0; i < kVPage / 16; ++i) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  __syncwarp();  // the zeroed pages are written before the arrival below releases them
  if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)__popc(okmask) * (uint32_t)kVPage);
  __syncwarp();
  if (ok) tma_load_5d(box, map, bar, 0, 0, 0, h, id);
}

// Each lane of a warp holds 64 contiguous output bytes of its own row (rows are
// 256 bytes to kilobytes apart in memory).  Store them 16 rows at a time through
// the warp's 1 KB staging area, so that 4 lanes write each row's 64 bytes
// together; the 16-byte pieces are XOR-swizzled by row against bank conflicts.
__device__ __forceinline__ void store_rows_coalesced(uint4 *stage, void *dst, bool ok, const uint4 (&v)[4],
                                                     int lane) {
  constexpr unsigned FULL = 0xffffffffu;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    if ((lane >> 4) == pass) {
      const int row = lane & 15;
#pragma unroll
      for (int i = 0; i < 4; ++i) stage[row * 4 + (i ^ (row & 3))] = v[i];
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int idx = lane + 32 * k;  // 64 pieces: row idx / 4, piece idx % 4
      const int row = idx >> 2, piece = idx & 3;
      const int src = pass * 16 + row;
      uint4 *d = reinterpret_cast<uint4 *>(__shfl_sync(FULL, reinterpret_cast<unsigned long long>(dst), src));
      const bool okr = __shfl_sync(FULL, ok ? 1 : 0, src) != 0;
      const uint4 w = stage[row * 4 + (piece ^ (row & 3))];
      if (okr) d[piece] = w;
    }
    __syncwarp();
  }
}

// ---- 8-bit pools: codes -> f16 operands ----------------------------------------

// f16 pair (lo in the low half) of two fp32 values, rounded to nearest, clamped
// to the finite range.
__device__ __forceinline__ uint32_t f16x2_satfinite(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// A row's scale s as the f16 pair sh + sl (sh = s rounded, sl = the remainder
// rounded: sh + sl = s to about 2^-22), both broadcast to f16x2.
struct ScaleH {
  __half2 hi, lo;
};
__device__ __forceinline__ ScaleH split_scale(float s) {
  const __half h = __float2half_rn(s);
  const __half l = __float2half_rn(s - __half2float(h));
  return {__half2half2(h), __half2half2(l)};
}

// Four codes of the word w as four f16 values code * s, in memory order.  The
// codes are exact in f16 (int8: the byte c + 128 placed in the low byte of
// the f16 1024 gives c + 1152 exactly, less 1152; E4M3: one exact conversion
// per pair), and code * s = fma(code, sh, code * sl) with a single rounding of
// a sum whose small term is exact to 2^-22 relative: code * s rounded once to
// f16, as through fp32, without leaving the f16 units.
template <int CODES>
__device__ __forceinline__ uint2 dequant4(uint32_t w, ScaleH s) {
  __half2 a, b;
  if constexpr (CODES == 1) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 bias = u32_as_h2(0xE480E480u);  // -1152, -1152
    a = __hadd2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4140u)), bias);
    b = __hadd2(u32_as_h2(__byte_perm(u, 0x64646464u, 0x4342u)), bias);
  } else {
    const __half2_raw ra = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
    const __half2_raw rb = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w >> 16), __NV_E4M3);
    a = *reinterpret_cast<const __half2 *>(&ra);
    b = *reinterpret_cast<const __half2 *>(&rb);
  }
  a = __hfma2(a, s.hi, __hmul2(a, s.lo));
  b = __hfma2(b, s.hi, __hmul2(b, s.lo));
  return make_uint2(h2_as_u32(a), h2_as_u32(b));
}

// One page (16 rows of 128 codes, row j at codes + 128 j) into f16: row j's
// dims 0..63 at out0 + 128 j and dims 64..127 at out1 + 128 j, the eight
// 16-byte pieces of each XOR-swizzled by j % 8 (the MMA operands' 128-byte
// swizzle), the values code * scale of the row (lane l < 16 holds the scale of
// row l in s).  Lane 8 p + 4 hh + jj converts dims 64 hh .. 64 hh + 63 of row
// 4 p + jj, visiting its four 16-code chunks from chunk (jj + 2 hh) % 4 on:
// with the swizzle, each quarter-warp's loads and stores hit 8 distinct 16-byte
// bank groups.  out1's rows are where the codes are: every lane of the warp
// loads its codes before any lane stores.  A row with its bit clear in `valid`
// (past the sequence, or the page not loaded) becomes zeros.  Straight-line,
// so that the sixteen conversions of a lane interleave.
template <int CODES>
__device__ __forceinline__ void convert_page(const uint8_t *codes, uint8_t *out0, uint8_t *out1, float s,
                                             uint32_t valid, int lane) {
  const int jj = lane & 3, hh = (lane >> 2) & 1, j = 4 * (lane >> 3) + jj;
  const ScaleH sj = split_scale(__shfl_sync(0xffffffffu, s, j));
  uint4 c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {  // c[i]: the 16 codes of chunk (i + jj + 2 hh) % 4 of this half-row
    const int ci = (i + jj + 2 * hh) & 3;
    c[i] = *reinterpret_cast<const uint4 *>(codes + j * 128 + hh * 64 + ci * 16);
  }
  __syncwarp();
  uint8_t *dst = (hh ? out1 : out0) + j * 128;
  const uint32_t keep = ((valid >> j) & 1) ? 0xffffffffu : 0u;  // zeros for a row outside the sequence
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ci = (i + jj + 2 * hh) & 3;
    const uint2 a = dequant4<CODES>(c[i].x, sj), b = dequant4<CODES>(c[i].y, sj);
    const uint2 e = dequant4<CODES>(c[i].z, sj), f = dequant4<CODES>(c[i].w, sj);
    *reinterpret_cast<uint4 *>(dst + (((2 * ci) ^ (j & 7)) << 4)) =
        make_uint4(a.x & keep, a.y & keep, b.x & keep, b.y & keep);
    *reinterpret_cast<uint4 *>(dst + (((2 * ci + 1) ^ (j & 7)) << 4)) =
        make_uint4(e.x & keep, e.y & keep, f.x & keep, f.y & keep);
  }
}

// Two pages at once (as convert_page each): every lane loads both pages'
// codes, then converts them, so the 32 conversions of a lane interleave.
template <int CODES>
__device__ __forceinline__ void convert_two_pages(const uint8_t *codes0, uint8_t *o00, uint8_t *o01, float s0,
                                                  uint32_t valid0, const uint8_t *codes1, uint8_t *o10,
                                                  uint8_t *o11, float s1, uint32_t valid1, int lane) {
  const int jj = lane & 3, hh = (lane >> 2) & 1, j = 4 * (lane >> 3) + jj;
  const ScaleH sa = split_scale(__shfl_sync(0xffffffffu, s0, j));
  const ScaleH sb = split_scale(__shfl_sync(0xffffffffu, s1, j));
  uint4 ca[4], cb[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ci = (i + jj + 2 * hh) & 3;
    ca[i] = *reinterpret_cast<const uint4 *>(codes0 + j * 128 + hh * 64 + ci * 16);
    cb[i] = *reinterpret_cast<const uint4 *>(codes1 + j * 128 + hh * 64 + ci * 16);
  }
  __syncwarp();
  uint8_t *da = (hh ? o01 : o00) + j * 128, *db = (hh ? o11 : o10) + j * 128;
  const uint32_t ka = ((valid0 >> j) & 1) ? 0xffffffffu : 0u, kb = ((valid1 >> j) & 1) ? 0xffffffffu : 0u;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int ci = (i + jj + 2 * hh) & 3;
    const uint2 a = dequant4<CODES>(ca[i].x, sa), b = dequant4<CODES>(ca[i].y, sa);
    const uint2 e = dequant4<CODES>(ca[i].z, sa), f = dequant4<CODES>(ca[i].w, sa);
    const uint2 a2 = dequant4<CODES>(cb[i].x, sb), b2 = dequant4<CODES>(cb[i].y, sb);
    const uint2 e2 = dequant4<CODES>(cb[i].z, sb), f2 = dequant4<CODES>(cb[i].w, sb);
    *reinterpret_cast<uint4 *>(da + (((2 * ci) ^ (j & 7)) << 4)) = make_uint4(a.x & ka, a.y & ka, b.x & ka, b.y & ka);
    *reinterpret_cast<uint4 *>(da + (((2 * ci + 1) ^ (j & 7)) << 4)) = make_uint4(e.x & ka, e.y & ka, f.x & ka, f.y & ka);
    *reinterpret_cast<uint4 *>(db + (((2 * ci) ^ (j & 7)) << 4)) =
        make_uint4(a2.x & kb, a2.y & kb, b2.x & kb, b2.y & kb);
    *reinterpret_cast<uint4 *>(db + (((2 * ci + 1) ^ (j & 7)) << 4)) =
        make_uint4(e2.x & kb, e2.y & kb, f2.x & kb, f2.y & kb);
  }
}

// bf16 bits of the largest magnitude in query row r of the Q tile (its two
// 64-dim halves at q + 128 r and q + kHalf + 128 r; the pieces are visited
// from a lane-dependent start so that a quarter-warp's loads hit distinct banks).
__device__ __forceinline__ uint32_t qrow_absmax_bf16(const uint8_t *q, int r, int lane) {
  uint32_t m = 0;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 w = *reinterpret_cast<const uint4 *>(q + hh * kHalf + r * 128 + (((i + lane) & 7) << 4));
      m = __vmaxu2(m, w.x & 0x7fff7fffu);  // magnitudes of finite bf16 values order as integers
      m = __vmaxu2(m, w.y & 0x7fff7fffu);
      m = __vmaxu2(m, w.z & 0x7fff7fffu);
      m = __vmaxu2(m, w.w & 0x7fff7fffu);
    }
  return max(m & 0xffffu, m >> 16);
}

// The 64 bf16 values of one half-row (at row, 128 bytes) rewritten in place as
// f16 of value * f (f a power of two; exact for results of at least 2^-17).
__device__ __forceinline__ void qrow_to_f16(uint8_t *row, float f, int lane) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint4 *pp = reinterpret_cast<uint4 *>(row + (((i + lane) & 7) << 4));
    uint4 w = *pp;
    uint32_t *u = reinterpret_cast<uint32_t *>(&w);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      u[k] = f16x2_satfinite(__uint_as_float(u[k] << 16) * f, __uint_as_float(u[k] & 0xffff0000u) * f);
    *pp = w;
  }
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// P = 2^(S * scale_log2 - m) for this thread's 64 keys of one tile (two
// 32-column chunks v[0], v[1]), unless `full` masked outside the row's visible
// keys (key kb + i of the half is visible when 0 <= kb + i <= span), written over
// the chunk's first 16 columns as pairs of the input dtype; with LO, the
// rounding remainder goes into the next 16.  Returns the row sum of P.
template <typename T, bool LO>
__device__ __forceinline__ float exp_pack_store(const uint32_t (&v)[2][32], uint32_t s_addr, float sl2, float m_ref,
                                                bool full, int kb, int span) {
  const float2 sl2v = make_float2(sl2, sl2), negm = make_float2(-m_ref, -m_ref);
  const float2 neg1 = make_float2(-1.f, -1.f);
  // the two chunks interleaved and four partial sums: short dependency chains
  float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  uint32_t pk[2][LO ? 32 : 16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const float2 sv = make_float2(__uint_as_float(v[cc][2 * j]), __uint_as_float(v[cc][2 * j + 1]));
      const float2 e = __ffma2_rn(sv, sl2v, negm);
      float2 pr = make_float2(ex2(e.x), ex2(e.y));
      if (!full) {
        const int key = kb + cc * 32 + 2 * j;
        pr.x = ((unsigned)key <= (unsigned)span) ? pr.x : 0.f;
        pr.y = ((unsigned)(key + 1) <= (unsigned)span) ? pr.y : 0.f;
      }
      float2 &acc = ls[(2 * j + cc) & 3];
      acc = __fadd2_rn(acc, pr);
      pk[cc][j] = Pack<T>::from_f2(pr.x, pr.y);
      if constexpr (LO) {
        const float2 lo = __ffma2_rn(Pack<T>::to_f2(pk[cc][j]), neg1, pr);  // P - P_hi, exact
        pk[cc][16 + j] = Pack<T>::from_f2(lo.x, lo.y);
      }
    }
  }
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    if constexpr (LO) {
      tc::st_32x32b_x32(s_addr + cc * 32, pk[cc]);
    } else {
      tc::st_32x32b_x16(s_addr + cc * 32, pk[cc]);
    }
  }
  const float2 t = __fadd2_rn(__fadd2_rn(ls[0], ls[1]), __fadd2_rn(ls[2], ls[3]));
  return t.x + t.y;
}

// The converter role over an 8-bit pool (loader warp lw of the CTA): warps
// 0 .. kKConv - 1 own the K pages wi, wi + kKConv, ... of every key tile, the
// others the V pages wi, wi + kVConv, ... (at most 3 per warp).  Per tile t:
// fetch tile t + 1's codes into the stage that tile t - 2 released (K: once
// its S was computed; V: once its P V product was done), so that no
// conversion waits for the tensor core's latest step; wait for tile t's
// codes, rewrite them as f16 rows in place, two pages per pass (K: page p's
// codes in the stage's upper 64-dim half where its rows' dims 64..127 go; V:
// in the upper half of the page's 4 KB); arrive on the tile's K / V barrier.  The scales of each
// lane's row are loaded with the codes, and the pages' block ids a tile
// before that.  Pages past the sequence are not fetched and their rows, like
// every row of a key >= ctx, become zeros; a block id outside the pool is
// reported and its page zeroed.  Returns false on a timed-out wait, after
// giving its copies in flight a bounded chance to land.
struct Fetch {
  float s[3];     // the scale of the lane's row in each of the warp's pages of the tile
  unsigned okm;   // bit k: page k was fetched
};
struct PageIds {
  int v[3];       // block id of each of the warp's pages of a tile (-1: past the sequence)
};
template <int CODES>
__device__ __forceinline__ bool convert_role(uint8_t *smem, Bars &bars, const CUtensorMap *kmap,
                                             const CUtensorMap *vmap, const PrefillParams &p, int c, int h,
                                             int kt0, int npages, int ntl, int ctx, const int32_t *bt, int lw,
                                             int lane) {
  const bool kside = lw < kKConv;
  const int wi = kside ? lw : lw - kKConv, nw = kside ? kKConv : kVConv;
  const CUtensorMap *map = kside ? kmap : vmap;
  const float *scales = kside ? p.k_scale : p.v_scale;
  uint64_t *cbar = kside ? bars.kc_full : bars.vc_full;  // codes landed
  uint64_t *dbar = kside ? bars.k_full : bars.v_full;    // f16 rows written
  uint64_t *fbar = kside ? bars.s_full : bars.pv_done;   // stage released
  uint8_t *ring = smem + (kside ? OFF_K : OFF_V);
  const int j = lane & 15;  // the row whose scale this lane holds in each page
  // page wi + nw k of tile t (k < 3, page < 8): its f16 rows, and where its codes land
  auto out0_of = [&](int st, int page) {
    return ring + st * 2 * kHalf + (kside ? page * kCodePage : page * kVPage);
  };
  auto codes_of = [&](int st, int page) { return out0_of(st, page) + (kside ? kHalf : kVPage / 2); };
  // Block ids of tile t's pages, read a tile before they are used (predicated
  // loads straight into the registers: nothing waits for them until then).
  auto ids_of = [&](int t) {
    PageIds r;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int page = wi + nw * k;
      const int pg = (kt0 + t) * 8 + page;
      r.v[k] = -1;
      if (t < ntl && page < 8 && pg < npages) r.v[k] = __ldg(bt + pg);
    }
    return r;
  };
  // Fetch tile t's codes (lane k < 3 issues page k's box) and the scale of this
  // lane's row in each page (from block 0 for a page not fetched, so that the
  // load is unconditional and nothing waits for it before the tile is converted).
  auto issue = [&](int t, const PageIds &ids) {
    const int st = t % kKStages;
    Fetch f;
    f.okm = 0;
    int my_id = -1;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int id = ids.v[k];
      const bool in = wi + nw * k < 8 && (kt0 + t) * 8 + wi + nw * k < npages;
      const bool ok = in && (unsigned)id < (unsigned)p.num_blocks;
      if (in && !ok && lane == 0) set_error(p.err, PA_ERR_RANGE, c);  // the error word reports the chunk
      f.s[k] = __ldg(scales + ((int64_t)(ok ? id : 0) * p.num_kv_heads + h) * kBlock + j);
      f.okm |= ok ? 1u << k : 0u;
      my_id = lane == k ? id : my_id;
    }
    if (lane == 0) mbar_arrive_expect_tx(&cbar[st], (uint32_t)__popc(f.okm) * (uint32_t)kCodePage);
    __syncwarp();
    if (lane < 3 && ((f.okm >> lane) & 1)) tma_load_4d(codes_of(st, wi + nw * lane), map, &cbar[st], 0, h, 0, my_id);
    return f;
  };
  Fetch fa{}, fb{};  // tiles t and t + 1
  bool ok = true;
  fa = issue(0, ids_of(0));
  PageIds idn = ids_of(1);  // the next tile to fetch
  int issued = 1;           // tiles whose codes this warp has fetched
  for (int t = 0; t < ntl; ++t) {
    const int st = t % kKStages;
    // tile t + 1's codes first, into the stage that tile t - 2 released: they
    // land while tile t is converted, so the conversions run back to back
    if (t + 1 < ntl) {
      if (t >= 2 && !mbar_wait(&fbar[(t - 2) % kKStages], ((t - 2) / kKStages) & 1)) {
        ok = false;
        break;
      }
      fb = issue(t + 1, idn);
      idn = ids_of(t + 2);
      issued = t + 2;
    }
    if (!mbar_wait(&cbar[st], (t / kKStages) & 1)) {
      ok = false;
      break;
    }
    {
      // pages 0 and 1 of the warp (every converter has at least two), then page 2 if any
      auto rows_valid = [&](int k, int page) {
        const int nrow = ((fa.okm >> k) & 1) ? ctx - ((kt0 + t) * 128 + page * 16) : 0;
        return nrow >= 16 ? 0xffffu : (nrow > 0 ? (1u << nrow) - 1u : 0u);
      };
      const int p0 = wi, p1 = wi + nw, p2 = wi + 2 * nw;
      uint8_t *a0 = out0_of(st, p0), *a1 = out0_of(st, p1);
      const int up = kside ? kHalf : kVPage / 2;
      convert_two_pages<CODES>(codes_of(st, p0), a0, a0 + up, fa.s[0], rows_valid(0, p0), codes_of(st, p1), a1,
                               a1 + up, fa.s[1], rows_valid(1, p1), lane);
      if (p2 < 8) {
        uint8_t *a2 = out0_of(st, p2);
        convert_page<CODES>(codes_of(st, p2), a2, a2 + up, fa.s[2], rows_valid(2, p2), lane);
      }
    }
    fence_proxy_async_smem();  // the generic writes reach the tensor core's reads
    __syncwarp();
    if (lane == 0) mbar_arrive(&dbar[st]);
    fa = fb;
  }
  if (!ok) {
    for (int t = issued - kKStages > 0 ? issued - kKStages : 0; t < issued; ++t)
      mbar_wait(&cbar[t % kKStages], (t / kKStages) & 1, kWaitLimitNs / 8);
  }
  return ok;
}

// Whether query tile mt of chunk c has rows: 1 yes, 0 none (the chunk is
// shorter), -1 the chunk's metadata is bad (reported by the caller).  Also its
// first row in q / out.
template <int G>
__device__ __forceinline__ int tile_rows(const PrefillParams &p, int c, int mt, int &row0) {
  constexpr int TQ = 128 / G;
  const int start = __ldg(p.chunk_starts + c), len = __ldg(p.chunk_lens + c), ctx = __ldg(p.context_lens + c);
  row0 = 0;
  for (int i = 0; i < c; ++i) row0 += __ldg(p.chunk_lens + i);
  if (len < 1 || len > p.max_chunk_len || start < 0 || ctx != start + len || ctx > p.max_blocks_per_seq * kBlock ||
      row0 + len > p.total_q_tokens)
    return -1;
  return mt * TQ < len ? 1 : 0;
}

// One query tile (chunk c, KV head h, query tile mt, which has rows: see
// tile_rows) computed by the whole CTA of kThreads threads, with the shared
// memory at smem (1024-aligned) and the 512 tensor-memory columns at tmem
// (allocated by the caller, or, when tmem_in is kTmemAllocHere, by this call
// beside the barriers' set-up and left to the caller to free from
// bars.tmem_base).  The tile's barriers are initialised on entry;
// with `reuse` they are invalidated before the return, which follows a
// CTA-wide barrier, so that the CTA may run another tile (the invalidation
// costs the last CTA about 0.6 µs, so a CTA of one tile skips it).  Returns false, in every thread, if a
// wait of any thread timed out (reported; asynchronous work of the tile was
// given a bounded chance to end).
// CODES: 0 = a 16-bit pool of the query dtype T; 1 = int8 codes, 2 = E4M3
// codes (kmap and vmap then address the code pools, one page of one KV head
// per box), the products computed in f16.
// RS / RO: the registers of the softmax warps and of the loader / converter
// and MMA warps inside the tile (2 x 128 x (RS + RO) <= 65536).
template <typename T, int G, int CODES, int RS = (CODES ? kRegsSoftmax8 : kRegsSoftmax),
          int RO = (CODES ? kRegsOther8 : kRegsOther)>
__device__ __forceinline__ bool prefill_tile(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                             const CUtensorMap &qmap, const CUtensorMap &omap,
                                             const PrefillParams &p, uint8_t *smem, uint32_t tmem_in, int c,
                                             int h, int mt, int row0, bool reuse) {
  constexpr int TQ = 128 / G;  // query tokens per tile
  using TC = typename std::conditional<CODES == 0, T, __half>::type;  // the MMA operand type (and P's)
  constexpr bool kBF16 = std::is_same<TC, __nv_bfloat16>::value;
  constexpr bool kQConv = CODES != 0 && std::is_same<T, __nv_bfloat16>::value;  // Q rewritten as f16
  constexpr uint32_t IDESC_S = tc::idesc_f16(kBF16, 128, 128, false);
  constexpr uint32_t IDESC_O = tc::idesc_f16(kBF16, 128, 128, true);
  constexpr unsigned FULL = 0xffffffffu;

  Bars &bars = *reinterpret_cast<Bars *>(smem + OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // No kernel of this library writes the chunk metadata or the block tables,
  // so they are read, and shared and tensor memory set up, while the previous
  // kernel may still run; only the loader warps, before their first copy of
  // Q, K or V, wait for it (every other warp consumes what the loaders fetch,
  // so its output stores also come after that wait).
  const int start = __ldg(p.chunk_starts + c), len = __ldg(p.chunk_lens + c), ctx = __ldg(p.context_lens + c);
  const int t0 = mt * TQ;
  const int last_key = min(start + t0 + TQ - 1, ctx - 1);  // largest key any row of the tile sees
  const int nkt = last_key / 128 + 1;
  const int kt_ctx = (ctx - 1) / 128;                       // key tile holding the sequence's last key
  const int npages = (ctx + kBlock - 1) / kBlock;
  const int32_t *bt = p.block_tables + (int64_t)c * p.max_blocks_per_seq;
  // Sliding window: the smallest key any row of the tile sees, the key tile
  // the loop starts at (tiles are counted from it: i = kt - kt0 indexes the
  // rings, the S buffers and the barrier phases) and the first page read.
  const int win = p.window;
  const int klo = (win > 0 && start + t0 - win + 1 > 0) ? start + t0 - win + 1 : 0;
  const int kt0 = klo / 128, pg0 = klo / kBlock, ntl = nkt - kt0;
  // Rows that see fewer than 128 keys average the rounding errors of too few
  // probabilities; they get the two-term P on the tiles where they occur: key
  // tile 0 for the tile's first rows, every tile under a window shorter than
  // 128.  Tiles i < lo_tiles (counted from kt0) take it.
  const int lo_tiles = (win > 0 && win < 128) ? ntl : (start + t0 < 127 ? 1 : 0);

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
    tma_prefetch_desc(&qmap);
    tma_prefetch_desc(&omap);
    mbar_init(&bars.q_full, 1);
    for (int b = 0; b < kKStages; ++b) {
      mbar_init(&bars.k_full[b], CODES ? kKConv : kLoadWarps);
      mbar_init(&bars.v_full[b], CODES ? kVConv : kLoadWarps);
      mbar_init(&bars.s_full[b], 1);
      mbar_init(&bars.p_full[b], kSoftmaxThreads);
      mbar_init(&bars.pv_done[b], 1);
      if constexpr (CODES != 0) {
        mbar_init(&bars.kc_full[b], kKConv);
        mbar_init(&bars.vc_full[b], kVConv);
      }
    }
    mbar_init(&bars.x_full, kSoftmaxThreads);
    mbar_init(&bars.drain, 1);
    if constexpr (kQConv) mbar_init(&bars.q_conv, kSoftmaxThreads);
    fence_mbar_init();
  }
  if (tmem_in == kTmemAllocHere && warp == kWarpMma) {  // (beside thread 0's set-up: one barrier for both)
    tc::tmem_alloc(&bars.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_in == kTmemAllocHere ? bars.tmem_base : tmem_in;
  bool timed_out = false;

  if (warp < kSoftmaxWarps) {
    static_assert(2 * 128 * (RS + RO) <= 65536, "register split fits the launch");
    regs_inc<RS>();
    regs_taken();
    // ---------------- softmax + epilogue (warps 0..7) ----------------
    const int quad = warp & 3, ch = warp >> 2;       // TMEM lane quarter, key half of every tile
    const int r = quad * 32 + lane;                  // tile row = TMEM lane
    const int tq = t0 + r / G;                       // query token within the chunk
    const int head = h * G + r % G;
    // visible keys of this row: rlo .. lim; kb0 = first key of this thread's
    // half of the loop's first tile, relative to rlo; span = lim - rlo
    const int lim = min(start + tq, ctx - 1);
    const int rlo = (win > 0 && start + tq - win + 1 > 0) ? start + tq - win + 1 : 0;
    const bool none = lim < rlo;  // a row past the chunk under a short window: no key at all
    const int kb0 = none ? -(1 << 30) : kt0 * 128 + ch * 64 - rlo, span = none ? 0 : lim - rlo;
    const int kt_last = kt_ctx - kt0;                // tile (from kt0) holding the sequence's last key
    const int zrow = ctx - kt_ctx * 128;             // its first row past the sequence
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const uint32_t o_self = tmem + lane_base + kColO + ch * 128;
    float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;
    if constexpr (kQConv) {
      // Row r of the bf16 query tile becomes f16 of q * 2^e, e putting the row's
      // largest magnitude in [2^14, 2^15) (clamped to [-110, 110]), which the
      // f16 range holds exactly; the row's scores are then S 2^e, so its
      // scale_log2 takes 2^-e.  Both threads of the row read both halves, wait
      // for each other, and rewrite their own half.
      const bool qok = mbar_wait(&bars.q_full, 0);
      const uint32_t amax = qok ? qrow_absmax_bf16(smem + OFF_Q, r, lane) : 0u;
      named_barrier(3, kSoftmaxThreads);  // every thread has read its row before any half is rewritten
      const int e = amax == 0 ? 0 : max(-110, min(110, 141 - (int)(amax >> 7)));
      if (qok) {
        qrow_to_f16(smem + OFF_Q + ch * kHalf + r * 128, __uint_as_float((uint32_t)(127 + e) << 23), lane);
        fence_proxy_async_smem();  // the generic writes reach the tensor core's reads
        mbar_arrive(&bars.q_conv);
      } else {
        timed_out = true;
      }
      sl2 *= __uint_as_float((uint32_t)(127 - e) << 23);
    }

    for (int kt = 0; kt < ntl && !timed_out; ++kt) {  // kt: tile index from kt0
      const int sb = kt & 1;
      if (!mbar_wait(&bars.s_full[kt % kKStages], (kt / kKStages) & 1)) {
        timed_out = true;
        break;
      }
      tc::fence_after_sync();
      const uint32_t s_addr = tmem + lane_base + sb * 128 + ch * 64;
      const int kb = kb0 + kt * 128;                 // first key of this thread's half, from rlo
      uint32_t v[2][32];
      tc::ld_32x32b_x32(s_addr, v[0]);
      tc::ld_32x32b_x32(s_addr + 32, v[1]);
      tc::wait_ld();
      const bool full = __all_sync(FULL, kb >= 0 && kb + 63 <= span);
      const bool first = (m_ref == -INFINITY);             // nothing accumulated for this row yet
      // The common tile (all keys visible, a reference maximum already set,
      // one-term P) computes P against the current reference without looking
      // for the tile's maximum first: while no P exceeds 2^8 the reference
      // holds, and a row sum of at most 2^8 proves that.  Only a row whose sum
      // exceeds it (rare) takes its maximum, and if that exceeds the reference
      // by more than 2^8, O and l are rescaled and P is computed again from the
      // scores still in registers.  Other tiles take the maximum first.
      // warp-uniform (the TMEM stores inside are warp-wide): a row whose window
      // or causal limit hid every key so far still has no reference maximum
      const bool common = kt >= lo_tiles && __all_sync(FULL, full && !first);
      float mx = -INFINITY, ls = 0.f;
      if (common) ls = exp_pack_store<TC, false>(v, s_addr, sl2, m_ref, true, kb, span);
      if (!common || ls > kRescaleSum) {  // per lane: the maximum of the visible scores
        if (full) {  // four independent chains of three-input maxima
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
      const float mc = mx * sl2;   // -inf if no key of this half is visible yet
      const bool need = !first && (mc > m_ref + kRescale);
      const bool redo = __any_sync(FULL, need);
      if (redo) {  // warp-uniform: the TMEM accesses below are warp-wide
        if (common) tc::wait_st();
        const float f = need ? ex2(m_ref - mc) : 1.f;
        if (need) {
          l *= f;
          m_ref = mc;
        }
        const int j = kt - 1;       // (kt >= 1 here) every earlier P V has landed in O
        if (!mbar_wait(&bars.pv_done[j % kVStages], (j / kVStages) & 1)) {
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
        // P in the input dtype (two terms where the tile needs them), over this half's S columns
        ls = (kt < lo_tiles) ? exp_pack_store<TC, true>(v, s_addr, sl2, m_ref, full, kb, span)
                             : exp_pack_store<TC, false>(v, s_addr, sl2, m_ref, full, kb, span);
      }
      l += ls;
      tc::wait_st();

      if (CODES == 0 && kt == kt_last) {  // (over 8-bit pools the converters write those rows as zeros)
        // value rows of keys >= ctx in this half (partial last page, pages past
        // the end); this half's P V product is the only one that reads them
        const int vb = kt % kVStages;
        if (!mbar_wait(&bars.v_full[vb], (kt / kVStages) & 1)) {
          timed_out = true;
          break;
        }
        const int z0 = max(zrow, ch * 64), z1 = ch * 64 + 64;
        uint8_t *vbase = smem + OFF_V + vb * 2 * kHalf;
        for (int idx = (warp & 3) * 32 + lane; idx < (z1 - z0) * 16; idx += kSoftmaxThreads / 2) {
          const int row = z0 + (idx >> 4), part = idx & 15;
          *reinterpret_cast<uint4 *>(vbase + (row >> 4) * kVPage + (part >> 3) * (kVPage / 2) + (row & 15) * 128 +
                                     (part & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc::fence_before_sync();
      // the P V batch waits on this barrier alone, so it must also imply that V landed
      if ((CODES != 0 || kt != kt_last) && !mbar_wait(&bars.v_full[kt % kVStages], (kt / kVStages) & 1)) {
        timed_out = true;
        break;
      }
      mbar_arrive(&bars.p_full[kt % kVStages]);
    }

    // The row's output, once P V of its last tile has landed and the two halves
    // have met.  The waits' outcome is made warp-uniform before the output
    // path, whose tensor-memory loads and row stores are warp-wide: a warp in
    // which any thread timed out stores nothing.
    bool ok = !timed_out;
    const int j = ntl - 1;
    if (ok) ok = mbar_wait(&bars.pv_done[j % kVStages], (j / kVStages) & 1);
    float2 *xm = reinterpret_cast<float2 *>(smem + OFF_X);
    if (ok) {
      tc::fence_after_sync();
      // merge the two halves of the row
      xm[ch * 128 + r] = make_float2(m_ref, l);
      mbar_arrive(&bars.x_full);
      ok = mbar_wait(&bars.x_full, 0);
    }
    ok = __all_sync(FULL, ok) != 0;
    if (!ok) timed_out = true;
    const bool tile_store = t0 + TQ <= len;
    if (ok) {
      const float2 other = xm[(1 - ch) * 128 + r];
      const float m0 = ch == 0 ? m_ref : other.x, l0 = ch == 0 ? l : other.y;
      const float m1 = ch == 0 ? other.x : m_ref, l1 = ch == 0 ? other.y : l;
      const float M = fmaxf(m0, m1);
      const float f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - M);
      const float f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - M);
      const float inv = 1.f / (l0 * f0 + l1 * f1);
      const float g0 = f0 * inv, g1 = f1 * inv;
      T *op = reinterpret_cast<T *>(p.out) + ((int64_t)(row0 + tq) * p.num_q_heads + head) * kHeadDim + ch * 64;
      const uint32_t o0 = tmem + lane_base + kColO + ch * 64, o1 = o0 + 128;
      // A query tile wholly inside its chunk leaves through one TMA store per
      // 64-dim half: each thread puts its row's 64 outputs into the (now idle)
      // Q buffer in the 128-byte swizzled layout the Q tile came in, which is
      // the out tensor's own tile shape.  A tile that runs past the chunk's
      // end (its last rows belong to the next chunk) stores row by row.
      uint8_t *otile = smem + OFF_Q + ch * kHalf;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t a[32], b[32];
        tc::ld_32x32b_x32(o0 + cc * 32, a);  // warp-wide; only rows of the chunk are stored
        tc::ld_32x32b_x32(o1 + cc * 32, b);
        tc::wait_ld();
        uint4 w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            y[e] = __uint_as_float(a[8 * i + e]) * g0 + __uint_as_float(b[8 * i + e]) * g1;
          w[i].x = Pack<T>::from_f2(y[0], y[1]);
          w[i].y = Pack<T>::from_f2(y[2], y[3]);
          w[i].z = Pack<T>::from_f2(y[4], y[5]);
          w[i].w = Pack<T>::from_f2(y[6], y[7]);
        }
        if (tile_store) {  // 16-byte piece cc * 4 + i of row r, XOR-swizzled by r % 8
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4 *>(otile + r * 128 + (((cc * 4 + i) ^ (r & 7)) << 4)) = w[i];
        } else {
          // warp-wide (every lane takes part); rows past the chunk are not stored
          store_rows_coalesced(reinterpret_cast<uint4 *>(smem + OFF_STAGE + warp * kStageBytes), op + cc * 32,
                               tq < len, w, lane);
        }
      }
    }
    if (tile_store) {  // every softmax thread joins the barrier of the TMA store, whatever it wrote
      fence_proxy_async_smem();  // the generic writes reach the TMA engine
      named_barrier(2, kSoftmaxThreads);
      if (threadIdx.x == 0 && !timed_out) {
        tma_store_3d(&omap, smem + OFF_Q, 0, h * G, row0 + t0);
        tma_store_3d(&omap, smem + OFF_Q + kHalf, 64, h * G, row0 + t0);
        bulk_commit_group();
        bulk_wait_group_all();  // before the CTA ends and its shared memory is reused
      }
    }
    regs_dec<128>();
  } else {
    // every loader and MMA warp runs this one decrease (setmaxnreg acts on whole warpgroups)
    regs_dec<RO>();
    if (warp != kWarpMma) {
      // ---------------- loader warps: each tile's K and V boxes, a seventh per warp ----------------
      const int lw = warp - kWarpLoad0;
      int32_t *sbt = reinterpret_cast<int32_t *>(smem + OFF_BT);
      const int cached = min(min(npages, nkt * 8) - pg0, kBtCache);
      for (int i = lw * 32 + lane; i < cached; i += kLoadWarps * 32) sbt[i] = __ldg(bt + pg0 + i);
      named_barrier(1, kLoadWarps * 32);  // the cached block ids are complete
      griddep_wait();                     // Q, K and V may come from the previous kernel
      if (lw == 0 && lane == 0) {
        mbar_arrive_expect_tx(&bars.q_full, 2 * kHalf);
        tma_load_3d(smem + OFF_Q, &qmap, &bars.q_full, 0, h * G, row0 + t0);
        tma_load_3d(smem + OFF_Q + kHalf, &qmap, &bars.q_full, 64, h * G, row0 + t0);
      }
      if constexpr (CODES != 0) {
        if (!convert_role<CODES>(smem, bars, &kmap, &vmap, p, c, h, kt0, npages, ntl, ctx, bt, lw, lane)) {
          timed_out = true;
          if (lw == 0) mbar_wait(&bars.q_full, 0, kWaitLimitNs / 8);
        }
      } else {
      // K boxes lw, lw + 7, lw + 14 and V pages (lw + 5) % 7, + 7: at most 4 boxes per warp and tile
      const int kb0 = lw, vb0 = (lw + 5) % kLoadWarps;
      int k_issued = 0, v_issued = 0;  // tiles whose K / V boxes this warp has issued
      for (int t = 0; t < ntl; ++t) {
        const int ks = t % kKStages, vs = t % kVStages;
        if (t >= kKStages && !mbar_wait(&bars.s_full[ks], ((t - kKStages) / kKStages) & 1)) {
          timed_out = true;
          break;
        }
        load_boxes(smem + OFF_K + ks * 2 * kHalf, &kmap, &bars.k_full[ks], kt0 + t, kb0, h, pg0, npages, sbt, bt, p,
                   c, lane);
        k_issued = t + 1;
        if (t >= kVStages && !mbar_wait(&bars.pv_done[vs], ((t - kVStages) / kVStages) & 1)) {
          timed_out = true;
          break;
        }
        load_vpages(smem + OFF_V + vs * 2 * kHalf, &vmap, &bars.v_full[vs], kt0 + t, vb0, h, pg0, npages, sbt, bt,
                    p, c, lane);
        v_issued = t + 1;
      }
      if (timed_out) {
        // Before the CTA ends (and its shared memory is handed to another CTA),
        // give this warp's copies still in flight a short, bounded chance to
        // land: the last tile of each stage it issued (each stage's barrier is
        // at most at that tile's phase).  A barrier that another warp left
        // short of its arrivals never completes; the wait then just ends.
        if (lw == 0) mbar_wait(&bars.q_full, 0, kWaitLimitNs / 8);
        for (int t = k_issued - kKStages > 0 ? k_issued - kKStages : 0; t < k_issued; ++t)
          mbar_wait(&bars.k_full[t % kKStages], (t / kKStages) & 1, kWaitLimitNs / 8);
        for (int t = v_issued - kVStages > 0 ? v_issued - kVStages : 0; t < v_issued; ++t)
          mbar_wait(&bars.v_full[t % kVStages], (t / kVStages) & 1, kWaitLimitNs / 8);
      }
      }
    } else {
      // ---------------- MMA issuer ----------------
      // The whole warp runs this loop (waits, barrier phases, descriptors), and
      // one elected lane issues each batch of MMAs and its commit: from a
      // warp-uniform loop the MMAs issue at the tensor core's own rate (32.7 ns
      // each at M = N = 128, K = 16) even while the softmax warps on the same
      // sub-partition are busy, where a loop run by one lane alone measured
      // 46-49 ns per MMA.
      // Descriptors are built once; a k-step or a ring stage only moves the start
      // address field (bits 0..13, address >> 4), so each MMA costs a 64-bit add.
      // Shared-memory offsets stay below 256 KB, so the field never carries over.
      // The tensor core queues only a few MMAs, so any latency between two
      // batches leaves it idle: the P barrier of the next P V batch is probed
      // without blocking right after the QK^T batch is issued; only a P that
      // really is not ready yet costs a (bounded) blocking wait.
      const bool leader = elect_one();
      auto wait_all = [&](uint64_t *bar, uint32_t parity) {  // warp-uniform result
        return __all_sync(0xffffffffu, mbar_wait(bar, parity)) != 0;
      };
      if (!wait_all(kQConv ? &bars.q_conv : &bars.q_full, 0)) timed_out = true;  // (Q rewritten as f16 first)
      const uint64_t qdesc = tc::desc_sw128(smem_u32(smem + OFF_Q), 16, 1024);
      const uint64_t kdesc0 = tc::desc_sw128(smem_u32(smem + OFF_K), 16, 1024);
      // V stages hold 8 pages of 4 KB: the dims 64..127 of a page 2 KB after its dims 0..63
      const uint64_t vdesc0 = tc::desc_sw128(smem_u32(smem + OFF_V), kVPage / 2, 1024);
      constexpr uint64_t kStageStep = (2 * kHalf) >> 4;   // one ring stage
      constexpr uint64_t kHalfStep = kHalf >> 4;          // the other 64-dim half
      bool pv_ok = false;                                  // P (and so V) of the next P V batch is ready
      for (int kt = 0; kt <= ntl && !timed_out; ++kt) {   // kt: tile index from kt0
        const int j = kt - 1, sj = j & 1;                  // the tile whose P V is issued in this iteration
        const int jv = j % kVStages;
        if (kt < ntl) {
          const int b = kt % kKStages, sb = kt & 1;
          if (!wait_all(&bars.k_full[b], (kt / kKStages) & 1)) {
            timed_out = true;
            break;
          }
          tc::fence_after_sync();
          const uint64_t kdesc = kdesc0 + (uint64_t)b * kStageStep;
          const uint32_t s_col = tmem + sb * 128;
          if (leader) {
            tc::mma_f16(s_col, qdesc, kdesc, IDESC_S, 0u);
  #pragma unroll
            for (int kk = 1; kk < 8; ++kk) {
              const uint64_t off = (uint64_t)((kk >> 2) * kHalfStep + (kk & 3) * 2);   // 16-element k-step
              tc::mma_f16(s_col, qdesc + off, kdesc + off, IDESC_S, 1u);
            }
            tc::commit(&bars.s_full[b]);
          }
          __syncwarp();
          pv_ok = kt >= 1 && __all_sync(0xffffffffu, mbar_test_wait(&bars.p_full[jv], (j / kVStages) & 1));
        } else {
          pv_ok = false;
        }
        if (kt >= 1) {  // O_half += P V of the previous tile: keys 0..63 into O_0, 64..127 into O_1
          if (!pv_ok && !wait_all(&bars.p_full[jv], (j / kVStages) & 1)) {
            timed_out = true;
            break;
          }
          tc::fence_after_sync();
          const uint64_t vdesc = vdesc0 + (uint64_t)jv * kStageStep;
          const uint32_t p_col = tmem + sj * 128;
          const uint32_t first = j > 0 ? 1u : 0u;
          if (leader) {
            if (j < lo_tiles) {
  #pragma unroll
              for (int kk = 0; kk < 8; ++kk) {  // 16-key step: V rows 16 kk .. 16 kk + 15, into O of key half kk / 4
                const uint32_t o_col = tmem + kColO + (kk >> 2) * 128;
                const uint32_t a_hi = p_col + 32 * (kk >> 1) + 8 * (kk & 1);
                const uint64_t bdesc = vdesc + (uint64_t)(kk * (kVPage >> 4));   // page kk
                tc::mma_f16_ts(o_col, a_hi, bdesc, IDESC_O, (kk & 3) > 0 ? 1u : first);
                tc::mma_f16_ts(o_col, a_hi + 16, bdesc, IDESC_O, 1u);
              }
            } else {
  #pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                const uint32_t o_col = tmem + kColO + (kk >> 2) * 128;
                const uint32_t a_hi = p_col + 32 * (kk >> 1) + 8 * (kk & 1);
                const uint64_t bdesc = vdesc + (uint64_t)(kk * (kVPage >> 4));   // page kk
                tc::mma_f16_ts(o_col, a_hi, bdesc, IDESC_O, (kk & 3) > 0 ? 1u : first);
              }
            }
            tc::commit(&bars.pv_done[jv]);
          }
          __syncwarp();
        }
      }
      if (timed_out) {
        // The MMAs already issued may still be writing TMEM (and reading
        // shared memory): one more commit tracks all of them; wait for it,
        // bounded, before the CTA frees its TMEM and ends.
        if (leader) tc::commit(&bars.drain);
        __syncwarp();
        mbar_wait(&bars.drain, 0, kWaitLimitNs / 8);
      }
    }
    regs_wait_taken();  // (the softmax warps hold their registers by now)
    regs_inc<128>();
  }
  if (timed_out) set_error(p.err, PA_ERR_TIMEOUT, c);
  tc::fence_before_sync();
  const bool any_timed_out = __syncthreads_or(timed_out) != 0;  // (the result is the same in every thread)
  tc::fence_after_sync();
  if (!reuse) return !any_timed_out;
  if (threadIdx.x == 0) {  // nobody waits on the tile's barriers any more: invalidate the ones set up above
    mbar_inval(&bars.q_full);
    for (int b = 0; b < kKStages; ++b) {
      mbar_inval(&bars.k_full[b]);
      mbar_inval(&bars.v_full[b]);
      mbar_inval(&bars.s_full[b]);
      mbar_inval(&bars.p_full[b]);
      mbar_inval(&bars.pv_done[b]);
      if constexpr (CODES != 0) {
        mbar_inval(&bars.kc_full[b]);
        mbar_inval(&bars.vc_full[b]);
      }
    }
    mbar_inval(&bars.x_full);
    mbar_inval(&bars.drain);
    if constexpr (kQConv) mbar_inval(&bars.q_conv);
  }
  __syncthreads();  // (the next tile's set-up comes after the invalidation)
  return !any_timed_out;
}

// One CTA per (query tile, KV head, chunk), heaviest first (last chunk, last
// query tile).
template <typename T, int G, int CODES = 0>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
               const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars &bars = *reinterpret_cast<Bars *>(smem + OFF_BAR);
  const int c = p.num_chunks - 1 - (int)blockIdx.z;
  const int h = blockIdx.y;
  const int mt = (int)gridDim.x - 1 - (int)blockIdx.x;
  int row0 = 0;
  const int rows = tile_rows<G>(p, c, mt, row0);
  if (rows <= 0) {
    if (rows < 0 && mt == 0 && h == 0 && threadIdx.x == 0) set_error(p.err, PA_ERR_RANGE, c);
    griddep_launch_dependents();
    return;
  }
  prefill_tile<T, G, CODES>(kmap, vmap, qmap, omap, p, smem, kTmemAllocHere, c, h, mt, row0, false);
  if ((threadIdx.x >> 5) == kWarpMma) tc::tmem_dealloc(bars.tmem_base, kTmemCols);
  griddep_launch_dependents();
}

}  // namespace
}  // namespace pa
