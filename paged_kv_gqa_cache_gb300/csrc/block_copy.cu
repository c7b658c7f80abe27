// Copy-on-write block copy for sm_103a (page "Модуль 12: Финальный проект:
// мини-движок инференса", qwen_serve/paged.py, SequenceCache._cow_copy: the
// new block receives the old block's K and V in every layer).
//
// A pure bit copy bound by HBM bandwidth: one CTA per (pair, layer, K or V)
// moves one block (16 slots x num_kv_heads x 128 16-bit values, 32 KB with 8
// KV heads) with 128-bit loads, eight in flight per thread before the first
// store.  The layer pools are separate allocations, so their base addresses
// travel in the kernel parameters (up to kCopyLayers per launch).
#include "pa_device.cuh"

namespace pa {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;

__global__ void __launch_bounds__(kCopyThreads) block_copy_kernel(const BlockCopyParams p) {
  griddep_wait();  // the pools may have been written by the previous kernel
  const int pair = blockIdx.x, layer = blockIdx.y, kv = blockIdx.z;
  const int src = __ldg(p.pairs + 2 * pair), dst = __ldg(p.pairs + 2 * pair + 1);
  if ((unsigned)src >= (unsigned)p.num_blocks || (unsigned)dst >= (unsigned)p.num_blocks) {
    if (layer == 0 && kv == 0 && threadIdx.x == 0) set_error(p.err, PA_ERR_RANGE, pair);
    griddep_launch_dependents();
    return;
  }
  uint4 *base = static_cast<uint4 *>(kv ? p.v[layer] : p.k[layer]);
  const uint4 *s = base + (int64_t)src * p.block_vecs;
  uint4 *d = base + (int64_t)dst * p.block_vecs;
  for (int i0 = threadIdx.x; i0 < p.block_vecs; i0 += kCopyThreads * kCopyUnroll) {
    uint4 r[kCopyUnroll];
#pragma unroll
    for (int j = 0; j < kCopyUnroll; ++j) {
      const int i = i0 + j * kCopyThreads;
      if (i < p.block_vecs) r[j] = s[i];
    }
#pragma unroll
    for (int j = 0; j < kCopyUnroll; ++j) {
      const int i = i0 + j * kCopyThreads;
      if (i < p.block_vecs) st_v4(d + i, r[j]);
    }
  }
  griddep_launch_dependents();
}

}  // namespace

cudaError_t launch_block_copy(const BlockCopyParams &p, int num_layers, int num_pairs, cudaStream_t stream) {
  return launch_pdl(block_copy_kernel, dim3(num_pairs, num_layers, 2), dim3(kCopyThreads), 0, stream, p);
}

}  // namespace pa
