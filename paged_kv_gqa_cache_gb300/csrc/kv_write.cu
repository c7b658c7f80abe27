// kv_cache_write for sm_103a: scatter the K/V rows of the step's new tokens
// into their pool slots (page "Модуль 12: Финальный проект: мини-движок
// инференса", qwen_serve/paged.py, PagedKVCache.write).
//
// A pure bit copy, bound by HBM bandwidth: each token row (num_kv_heads x 128
// 16-bit values, 2 KB for 8 KV heads) is read once from k/v and written once
// into slot slot_mapping[t] of the pool, with 128-bit coalesced loads and
// stores.  Consecutive threads take consecutive 16-byte vectors of one row, so
// every warp moves whole 512-byte runs.
#include "pa_device.cuh"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) kv_write_kernel(const WriteParams p) {
  // The next kernel (a decode) may start its set-up at once, beside the tail
  // of the kernel before this one; it still waits for this grid to complete,
  // which comes after that kernel has completed, before it reads anything
  // but what it is allowed to read early.
  griddep_launch_dependents();
  griddep_wait();
  const int64_t total = (int64_t)p.num_tokens * p.row_vecs;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const int t = (int)(i / p.row_vecs);
    const int vi = (int)(i - (int64_t)t * p.row_vecs);
    const int64_t slot = __ldg(p.slots + t);
    if (slot < 0 || slot >= p.num_slots) {
      if (vi == 0) set_error(p.err, PA_ERR_RANGE, t);
      continue;
    }
    const uint4 kv = ld_nc_v4(static_cast<const uint4 *>(p.k) + i);
    const uint4 vv = ld_nc_v4(static_cast<const uint4 *>(p.v) + i);
    st_v4(static_cast<uint4 *>(p.k_cache) + slot * p.row_vecs + vi, kv);
    st_v4(static_cast<uint4 *>(p.v_cache) + slot * p.row_vecs + vi, vv);
  }
}

// Quantising write into an int8 pool ("Модуль 04: KV-кэш и арифметика памяти",
// section 5, KV8Cache.write): for each new token and KV head, and for K and V
// separately, scale = max |x| / 127 + 1e-8 and code = clip(rint(x / scale),
// -127, 127), every step in fp32 rounded to nearest (an IEEE division, ties of
// rint to even), so the codes are exactly the ones the method defines.  One
// warp per (token, KV head) row of 128 values: lane j owns values 4j .. 4j + 3,
// the row maximum is a warp reduction, each lane stores its 4 codes as one
// 32-bit word and lane 0 stores the scale.
template <typename T, bool F8>
__global__ void __launch_bounds__(256) kv_write_q8_kernel(const WriteQ8Params p) {
  griddep_launch_dependents();  // as the 16-bit write: the next kernel may start its set-up at once
  griddep_wait();
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)p.num_tokens * p.num_kv_heads;
  const int64_t wstride = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += wstride) {
    const int t = (int)(r / p.num_kv_heads), h = (int)(r % p.num_kv_heads);
    const int64_t slot = __ldg(p.slots + t);
    if (slot < 0 || slot >= p.num_slots) {
      if (h == 0 && lane == 0) set_error(p.err, PA_ERR_RANGE, t);
      continue;
    }
    const int64_t si = ((slot >> 4) * p.num_kv_heads + h) * kBlock + (slot & 15);
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
      const uint2 u = __ldg(reinterpret_cast<const uint2 *>(pass == 0 ? p.k : p.v) + r * (kHeadDim / 4) + lane);
      const float2 a = Pack<T>::to_f2(u.x), b = Pack<T>::to_f2(u.y);
      float amax = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, off));
      const float scale = __fadd_rn(__fdiv_rn(amax, F8 ? 448.f : 127.f), 1e-8f);
      const float x[4] = {a.x, a.y, b.x, b.y};
      uint32_t word = 0;
      if constexpr (F8) {  // the nearest E4M3 value, ties to even (|x / scale| <= 448 by construction)
#pragma unroll
        for (int e = 0; e < 4; e += 2) {
          const __nv_fp8x2_storage_t c2 = __nv_cvt_float2_to_fp8x2(
              make_float2(__fdiv_rn(x[e], scale), __fdiv_rn(x[e + 1], scale)), __NV_SATFINITE, __NV_E4M3);
          word |= (uint32_t)c2 << (8 * e);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float c = fminf(fmaxf(rintf(__fdiv_rn(x[e], scale)), -127.f), 127.f);
          word |= ((uint32_t)(int)c & 0xffu) << (8 * e);
        }
      }
      int8_t *dst = pass == 0 ? p.k_cache : p.v_cache;
      reinterpret_cast<uint32_t *>(dst + (slot * p.num_kv_heads + h) * kHeadDim)[lane] = word;
      if (lane == 0) (pass == 0 ? p.k_scale : p.v_scale)[si] = scale;
    }
  }
}

}  // namespace

cudaError_t launch_kv_write_q8(const WriteQ8Params &p, int dtype, bool f8, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.num_tokens * p.num_kv_heads;
  int64_t grid = (rows + 7) / 8;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  const dim3 g((unsigned)grid), b(256);
  if (f8)
    return dtype == PA_BF16 ? launch_pdl(kv_write_q8_kernel<__nv_bfloat16, true>, g, b, 0, stream, p)
                            : launch_pdl(kv_write_q8_kernel<__half, true>, g, b, 0, stream, p);
  return dtype == PA_BF16 ? launch_pdl(kv_write_q8_kernel<__nv_bfloat16, false>, g, b, 0, stream, p)
                          : launch_pdl(kv_write_q8_kernel<__half, false>, g, b, 0, stream, p);
}

cudaError_t launch_kv_write(const WriteParams &p, cudaStream_t stream) {
  const int64_t total = (int64_t)p.num_tokens * p.row_vecs;
  int64_t grid = (total + 255) / 256;
  const int64_t cap = (int64_t)sm_count() * 8;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  return launch_pdl(kv_write_kernel, dim3((unsigned)grid), dim3(256), 0, stream, p);
}

}  // namespace pa
