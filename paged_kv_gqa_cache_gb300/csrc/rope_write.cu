// q/k RMSNorm + rotary embedding fused into the KV write, for sm_103a (page
// "Модуль 12: Финальный проект: мини-движок инференса", qwen_serve/model.py:
// rms_norm, _rotate_half, apply_rope and their use in Qwen3Model.forward before
// PagedKVCache.write; page "Модуль 04: KV-кэш и арифметика памяти", section 4:
// the key is rotated to its absolute position before it is stored).
//
// For each new token t at absolute position positions[t]:
//   q_out[t][g]        = rope(rms_norm(q[t][g], q_weight))   for every query head g,
//   pool slot of t, K  = rope(rms_norm(k[t][h], k_weight))   for every KV head h,
//   pool slot of t, V  = v[t][h].
// One pass over the step's q/k/v instead of a norm pass, a rotation pass and a
// copy: HBM-bound.  A warp takes four head rows of one token at a time (128
// values per row, 4 per lane, 8-byte loads and stores; all loads issued before
// the first use); the rotation pairs dims i and i + 64, i.e. lanes l and
// l ^ 16.
//
// Rounding follows the page's precision: the mean of squares and the
// reciprocal square root are fp32, every other step a 16-bit tensor operation
// (its fp32 result, exact for a product of two 16-bit values, rounded once to
// the 16-bit format, ties to even).  The fp32 mean is the one nearest the
// exact mean: the squares of 16-bit values are exact in fp32 and are summed as
// an unevaluated pair hi + lo of fp32 values with error-free additions
// (Knuth's two-sum, then Dekker's fast two-sum to renormalise), which is exact
// while the sum spans at most ~47 bits (for bf16 rows, squares within a factor
// 2^24 of each other) and otherwise off by far less than half an fp32 ulp;
// fp64 would do the same at a fraction of the speed on this part.  The
// reciprocal square root is the correctly rounded one.  Explicit
// round-to-nearest intrinsics keep the compiler from fusing or reordering.
#include "pa_device.cuh"

namespace pa {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kRopeThreads = 256;
constexpr int kRowsPerUnit = 4;  // head rows of one token per warp step

// Error-free fp32 additions: s + e == a + b exactly (two-sum: any a, b; fast
// two-sum: |a| >= |b| or a == 0).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

// hi + lo += x, renormalised so that hi = fl(hi + lo).
__device__ __forceinline__ void pair_add(float &hi, float &lo, float xhi, float xlo) {
  float s, e;
  two_sum(hi, xhi, s, e);
  fast_two_sum(s, __fadd_rn(__fadd_rn(lo, xlo), e), hi, lo);
}

// Packed 16-bit products and sums, each the exact result rounded once to the
// 16-bit format (ties to even) — a 16-bit tensor operation.  For a sum this
// equals rounding the fp32 sum to 16 bits: two 16-bit values add exactly in
// fp32 unless their exponents differ by more than 13 bits, and then the
// smaller is below half a 16-bit ulp of the larger either way.
template <typename T>
struct Packed;
template <>
struct Packed<__nv_bfloat16> {
  using V = __nv_bfloat162;
};
template <>
struct Packed<__half> {
  using V = __half2;
};
template <typename T>
__device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
  using V = typename Packed<T>::V;
  const V r = __hmul2_rn(*reinterpret_cast<const V *>(&a), *reinterpret_cast<const V *>(&b));
  return *reinterpret_cast<const uint32_t *>(&r);
}
template <typename T>
__device__ __forceinline__ uint32_t add2(uint32_t a, uint32_t b) {
  using V = typename Packed<T>::V;
  const V r = __hadd2_rn(*reinterpret_cast<const V *>(&a), *reinterpret_cast<const V *>(&b));
  return *reinterpret_cast<const uint32_t *>(&r);
}

// inv = rsqrt(mean(x^2) + eps) in fp32 for the 4 rows of a unit (this lane's
// 4 values of each in raw[i]).  The fp32 mean is the one nearest the exact
// mean (pair sums, see above).  Reduced as a transpose: at the first butterfly
// level lanes 0..15 keep rows 0, 1 and lanes 16..31 rows 2, 3, at the second
// each lane keeps one row, then a plain butterfly over 8 lanes; lane 8 i ends
// with row i, computes its inverse square root and broadcasts it.
template <typename T>
__device__ __forceinline__ void rows_rsqrt4(const uint2 (&raw)[4], float eps, int lane, float (&inv)[4]) {
  float hi[4], lo[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a = Pack<T>::to_f2(raw[i].x), b = Pack<T>::to_f2(raw[i].y);
    // squares of 16-bit values are exact in fp32; the local pair is renormalised at the first level below
    hi[i] = __fmul_rn(a.x, a.x);
    lo[i] = 0.f;
    const float sq[3] = {__fmul_rn(a.y, a.y), __fmul_rn(b.x, b.x), __fmul_rn(b.y, b.y)};
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      float sum, err;
      two_sum(hi[i], sq[k], sum, err);
      hi[i] = sum;
      lo[i] = __fadd_rn(lo[i], err);
    }
  }
  const bool up16 = lane & 16, up8 = lane & 8;
  // level 16: keep rows (0, 1) below lane 16, (2, 3) above; send the other two
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float shi = up16 ? hi[i] : hi[i + 2], slo = up16 ? lo[i] : lo[i + 2];
    const float rhi = __shfl_xor_sync(FULL, shi, 16), rlo = __shfl_xor_sync(FULL, slo, 16);
    float khi = up16 ? hi[i + 2] : hi[i], klo = up16 ? lo[i + 2] : lo[i];
    pair_add(khi, klo, rhi, rlo);
    hi[i] = khi;  // kept row (i, or i + 2 above lane 16), now in slot i
    lo[i] = klo;
  }
  // level 8: keep slot 0 where lane bit 3 is clear, slot 1 where set
  float h = up8 ? hi[1] : hi[0], l = up8 ? lo[1] : lo[0];
  {
    const float shi = up8 ? hi[0] : hi[1], slo = up8 ? lo[0] : lo[1];
    const float rhi = __shfl_xor_sync(FULL, shi, 8), rlo = __shfl_xor_sync(FULL, slo, 8);
    pair_add(h, l, rhi, rlo);
  }
#pragma unroll
  for (int off = 4; off > 0; off >>= 1) {
    const float rhi = __shfl_xor_sync(FULL, h, off), rlo = __shfl_xor_sync(FULL, l, off);
    pair_add(h, l, rhi, rlo);
  }
  // lane 8 i now holds row i: rows 0, 1 below lane 16 (slot by bit 3), rows 2, 3 above
  const float var = __fmul_rn(__fadd_rn(h, l), 1.f / kHeadDim);  // a power-of-two scaling: exact
  const float mine = __frsqrt_rn(__fadd_rn(var, eps));
#pragma unroll
  for (int i = 0; i < 4; ++i) inv[i] = __shfl_sync(FULL, mine, 8 * i);
}

// One head row after its inverse RMS: y = x inv (fp32, rounded to 16 bits),
// z = y w, then out = z cos + rotate_half(z) sin, rotate_half(z)[i] =
// -z[i + 64] (i < 64), z[i - 64] (i >= 64); this lane holds dims 4 lane ..
// 4 lane + 3, and dims i and i + 64 sit on lanes l and l ^ 16.
template <typename T>
__device__ __forceinline__ uint2 norm_rope_row(uint2 raw, float inv, uint2 wr, uint2 cr, uint2 sr, int lane) {
  const float2 x01 = Pack<T>::to_f2(raw.x), x23 = Pack<T>::to_f2(raw.y);
  const uint32_t y01 = Pack<T>::from_f2(__fmul_rn(x01.x, inv), __fmul_rn(x01.y, inv));
  const uint32_t y23 = Pack<T>::from_f2(__fmul_rn(x23.x, inv), __fmul_rn(x23.y, inv));
  const uint32_t z01 = mul2<T>(y01, wr.x), z23 = mul2<T>(y23, wr.y);
  const uint32_t neg = lane < 16 ? 0x80008000u : 0u;  // rotate_half's sign, on both halves of a pair
  const uint32_t p01 = __shfl_xor_sync(FULL, z01, 16) ^ neg, p23 = __shfl_xor_sync(FULL, z23, 16) ^ neg;
  uint2 out;
  out.x = add2<T>(mul2<T>(z01, cr.x), mul2<T>(p01, sr.x));
  out.y = add2<T>(mul2<T>(z23, cr.y), mul2<T>(p23, sr.y));
  return out;
}

// A warp takes kRowsPerUnit consecutive head rows of one token per step (the
// token's rows are its Hq query heads, then its Hkv key heads, then its Hkv
// value heads), issuing every load of the unit before the first use so that
// their latencies overlap.
template <typename T>
__global__ void __launch_bounds__(kRopeThreads) rope_write_kernel(const RopeWriteParams p) {
  griddep_wait();  // q/k/v may be the previous kernel's output; the pool may be read by it
  const int lane = threadIdx.x & 31;
  const int hq = p.num_q_heads, hkv = p.num_kv_heads;
  const int rows_per_token = hq + 2 * hkv;
  const int units_per_token = (rows_per_token + kRowsPerUnit - 1) / kRowsPerUnit;
  const int units = p.num_tokens * units_per_token;  // < 2^31 (checked on the host)
  const int nwarps = (int)(gridDim.x * kRopeThreads) >> 5;
  const uint2 wq = *reinterpret_cast<const uint2 *>(static_cast<const T *>(p.q_weight) + 4 * lane);
  const uint2 wk = *reinterpret_cast<const uint2 *>(static_cast<const T *>(p.k_weight) + 4 * lane);

  // the unit (token t, first row j0): its rows, position and slot; the rows' loads
  // do not depend on the position or slot
  auto fetch = [&](int t, int j0, uint2 (&raw)[kRowsPerUnit], int &pos, int64_t &slot) {
    pos = __ldg(p.positions + t);
    slot = __ldg(p.slots + t);
#pragma unroll
    for (int i = 0; i < kRowsPerUnit; ++i) {
      const int j = j0 + i;
      raw[i] = make_uint2(0, 0);
      if (j < rows_per_token) {
        const T *src = j < hq ? static_cast<const T *>(p.q) + ((int64_t)t * hq + j) * kHeadDim
                       : j < hq + hkv ? static_cast<const T *>(p.k) + ((int64_t)t * hkv + j - hq) * kHeadDim
                                      : static_cast<const T *>(p.v) + ((int64_t)t * hkv + j - hq - hkv) * kHeadDim;
        raw[i] = *reinterpret_cast<const uint2 *>(src + 4 * lane);
      }
    }
  };
  // software pipeline: the next unit's loads are in flight while this one is computed.
  // Unit u is (token u / units_per_token, group u % units_per_token); the warp's
  // units advance by nwarps, tracked as a token step and a group step.
  int u = (int)((blockIdx.x * kRopeThreads) >> 5) + (int)(threadIdx.x >> 5);
  const int dt = nwarps / units_per_token, dg = nwarps - dt * units_per_token;
  int t_next = u / units_per_token, g_next = u - t_next * units_per_token;
  uint2 raw[kRowsPerUnit], raw_next[kRowsPerUnit];
  int pos = 0, pos_next = 0;
  int64_t slot = 0, slot_next = 0;
  if (u < units) fetch(t_next, g_next * kRowsPerUnit, raw_next, pos_next, slot_next);
  for (; u < units; u += nwarps) {
#pragma unroll
    for (int i = 0; i < kRowsPerUnit; ++i) raw[i] = raw_next[i];
    pos = pos_next;
    slot = slot_next;
    const int t = t_next, j0 = g_next * kRowsPerUnit;
    t_next += dt;
    g_next += dg;
    if (g_next >= units_per_token) {
      g_next -= units_per_token;
      ++t_next;
    }
    if (u + nwarps < units) fetch(t_next, g_next * kRowsPerUnit, raw_next, pos_next, slot_next);
    const bool ok = pos >= 0 && pos < p.max_position && slot >= 0 && slot < p.num_slots;
    const int64_t prow = (int64_t)(ok ? pos : 0) * kHeadDim + 4 * lane;
    const uint2 cr = *reinterpret_cast<const uint2 *>(static_cast<const T *>(p.cos_table) + prow);
    const uint2 sr = *reinterpret_cast<const uint2 *>(static_cast<const T *>(p.sin_table) + prow);
    if (!ok) {  // warp-uniform; nothing of this token is written
      if (j0 == 0 && lane == 0) set_error(p.err, PA_ERR_RANGE, t);
      continue;
    }
    float inv[kRowsPerUnit];
    if (j0 < hq + hkv) rows_rsqrt4<T>(raw, p.eps, lane, inv);  // warp-uniform: the unit has q or k rows
#pragma unroll
    for (int i = 0; i < kRowsPerUnit; ++i) {
      const int j = j0 + i;
      if (j >= rows_per_token) break;
      T *dst;
      uint2 out;
      if (j < hq) {
        dst = static_cast<T *>(p.q_out) + ((int64_t)t * hq + j) * kHeadDim;
        out = norm_rope_row<T>(raw[i], inv[i], wq, cr, sr, lane);
      } else if (j < hq + hkv) {
        dst = static_cast<T *>(p.k_cache) + (slot * hkv + j - hq) * kHeadDim;
        out = norm_rope_row<T>(raw[i], inv[i], wk, cr, sr, lane);
      } else {  // a value row: stored unchanged
        dst = static_cast<T *>(p.v_cache) + (slot * hkv + j - hq - hkv) * kHeadDim;
        out = raw[i];
      }
      *reinterpret_cast<uint2 *>(dst + 4 * lane) = out;
    }
  }
  griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_rope_write(const RopeWriteParams &p, int dtype, cudaStream_t stream) {
  const int64_t units = (int64_t)p.num_tokens *
                       ((p.num_q_heads + 2 * p.num_kv_heads + kRowsPerUnit - 1) / kRowsPerUnit);
  int64_t ctas = (units + kRopeThreads / 32 - 1) / (kRopeThreads / 32);
  const int64_t cap = (int64_t)sm_count() * 4;  // one wave (4 CTAs of 8 warps fit per SM), then grid-stride
  if (ctas > cap) ctas = cap;
  if (dtype == PA_BF16)
    return launch_pdl(rope_write_kernel<__nv_bfloat16>, dim3((unsigned)ctas), dim3(kRopeThreads), 0, stream, p);
  return launch_pdl(rope_write_kernel<__half>, dim3((unsigned)ctas), dim3(kRopeThreads), 0, stream, p);
}

}  // namespace pa
