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
// released after the PV product.  Three loader warps fill both rings, each
// issuing a third of every tile's 24 boxes from parallel lanes: the TMA engine
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
// Warps 8..10 load Q, K and V, warp 11 owns TMEM and issues the
// MMAs (one thread); mbarriers hand tiles between the roles and every wait is
// bounded.  Keys above the diagonal are masked per element on the tiles that
// cross it (a warp-uniform test picks the unmasked path elsewhere) and never
// loaded past the tile holding the tile's last query.  Value rows past the
// sequence's last key are zeroed in shared memory before the PV product so that
// a zero probability never meets a non-finite value.
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
template <int N>
__device__ __forceinline__ void regs_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void regs_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
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
  uint32_t tmem_base;
};

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

template <typename T, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
               const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
               const PrefillParams p) {
  constexpr int TQ = 128 / G;  // query tokens per tile
  constexpr bool kBF16 = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t IDESC_S = tc::idesc_f16(kBF16, 128, 128, false);
  constexpr uint32_t IDESC_O = tc::idesc_f16(kBF16, 128, 128, true);
  constexpr unsigned FULL = 0xffffffffu;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  Bars &bars = *reinterpret_cast<Bars *>(smem + OFF_BAR);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // No kernel of this library writes the chunk metadata or the block tables,
  // so they are read, and shared and tensor memory set up, while the previous
  // kernel may still run; only the loader warps, before their first copy of
  // Q, K or V, wait for it (every other warp consumes what the loaders fetch,
  // so its output stores also come after that wait).

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
      mbar_init(&bars.k_full[b], kLoadWarps);
      mbar_init(&bars.v_full[b], kLoadWarps);
      mbar_init(&bars.s_full[b], 1);
      mbar_init(&bars.p_full[b], kSoftmaxThreads);
      mbar_init(&bars.pv_done[b], 1);
    }
    mbar_init(&bars.x_full, kSoftmaxThreads);
    mbar_init(&bars.drain, 1);
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

  if (warp < kSoftmaxWarps) {
    regs_inc<kRegsSoftmax>();
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
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY, l = 0.f;

    for (int kt = 0; kt < ntl; ++kt) {               // kt: tile index from kt0
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
      if (common) ls = exp_pack_store<T, false>(v, s_addr, sl2, m_ref, true, kb, span);
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
        ls = (kt < lo_tiles) ? exp_pack_store<T, true>(v, s_addr, sl2, m_ref, full, kb, span)
                             : exp_pack_store<T, false>(v, s_addr, sl2, m_ref, full, kb, span);
      }
      l += ls;
      tc::wait_st();

      if (kt == kt_last) {
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
      if (kt != kt_last && !mbar_wait(&bars.v_full[kt % kVStages], (kt / kVStages) & 1)) {
        timed_out = true;
        break;
      }
      mbar_arrive(&bars.p_full[kt % kVStages]);
    }

    if (!timed_out) {
      const int j = ntl - 1;
      if (mbar_wait(&bars.pv_done[j % kVStages], (j / kVStages) & 1)) {
        tc::fence_after_sync();
        // merge the two halves of the row
        float2 *xm = reinterpret_cast<float2 *>(smem + OFF_X);
        xm[ch * 128 + r] = make_float2(m_ref, l);
        mbar_arrive(&bars.x_full);
        if (mbar_wait(&bars.x_full, 0)) {
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
          const bool tile_store = t0 + TQ <= len;
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
          if (tile_store) {
            fence_proxy_async_smem();  // the generic writes reach the TMA engine
            named_barrier(2, kSoftmaxThreads);
            if (threadIdx.x == 0) {
              tma_store_3d(&omap, smem + OFF_Q, 0, h * G, row0 + t0);
              tma_store_3d(&omap, smem + OFF_Q + kHalf, 64, h * G, row0 + t0);
              bulk_commit_group();
              bulk_wait_group_all();  // before the CTA ends and its shared memory is reused
            }
          }
        } else {
          timed_out = true;
        }
      } else {
        timed_out = true;
      }
    }
    regs_dec<128>();
  } else {
    // every loader and MMA warp runs this one decrease (setmaxnreg acts on whole warpgroups)
    regs_dec<kRegsOther>();
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
      if (!wait_all(&bars.q_full, 0)) timed_out = true;
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
    regs_inc<128>();
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
