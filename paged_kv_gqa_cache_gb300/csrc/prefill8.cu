// Chunked prefill over 8-bit pools on the tcgen05 tensor cores: the per-tile
// kernel of prefill_kernel.cuh with its converter warps (CODES = 1: int8,
// 2: E4M3), one CTA per query tile and KV head.
#include "prefill_kernel.cuh"

namespace pa {
namespace {

template <typename T, int G, int CODES>
cudaError_t launch_codes(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                         const CUtensorMap &qmap, const CUtensorMap &omap, cudaStream_t stream) {
  static KernelSetup setup;
  cudaError_t e = kernel_setup(setup, prefill_kernel<T, G, CODES>, SMEM_BYTES, kThreads, nullptr);
  if (e != cudaSuccess) return e;
  constexpr int TQ = 128 / G;
  dim3 grid((p.max_chunk_len + TQ - 1) / TQ, p.num_kv_heads, p.num_chunks);
  return launch_pdl(prefill_kernel<T, G, CODES>, grid, dim3(kThreads), SMEM_BYTES, stream, kmap, vmap, qmap, omap,
                    p);
}

template <typename T, int CODES>
cudaError_t launch_group(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                         const CUtensorMap &qmap, const CUtensorMap &omap, int group, cudaStream_t stream) {
  switch (group) {
    case 1: return launch_codes<T, 1, CODES>(p, kmap, vmap, qmap, omap, stream);
    case 2: return launch_codes<T, 2, CODES>(p, kmap, vmap, qmap, omap, stream);
    case 4: return launch_codes<T, 4, CODES>(p, kmap, vmap, qmap, omap, stream);
    case 8: return launch_codes<T, 8, CODES>(p, kmap, vmap, qmap, omap, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_prefill8(const PrefillParams &p, const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const CUtensorMap &qmap, const CUtensorMap &omap, int dtype, int group, bool f8,
                               cudaStream_t stream) {
  if (p.window != 0 || p.ws_counters) return cudaErrorInvalidValue;
  if (dtype == PA_BF16)
    return f8 ? launch_group<__nv_bfloat16, 2>(p, kmap, vmap, qmap, omap, group, stream)
              : launch_group<__nv_bfloat16, 1>(p, kmap, vmap, qmap, omap, group, stream);
  return f8 ? launch_group<__half, 2>(p, kmap, vmap, qmap, omap, group, stream)
            : launch_group<__half, 1>(p, kmap, vmap, qmap, omap, group, stream);
}

}  // namespace pa
