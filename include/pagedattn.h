/*
 * libpagedattn — GQA attention over a paged KV cache, for GB300 (sm_103a).
 *
 * The operations follow two course pages:
 *   [P1] "Модуль 12: Финальный проект: мини-движок инференса" (LLM Inference
 *        Systems course): task 12.1 and the qwen_serve/paged.py listing
 *        (PagedKVCache: pool layout, write, read) and the qwen_serve/model.py
 *        listing (Qwen3Model.forward: GQA attention over the cached prefix,
 *        causal mask on absolute positions for multi-token steps).
 *   [P2] "Модуль 04: KV-кэш и арифметика памяти": section 1 (the attention
 *        output over cached K/V), section 3.4 (chunked prefill keeps its KV
 *        between chunks), task 04.1 (positions belong to the caller; the mask
 *        compares absolute positions).
 *
 * Conventions for every call:
 *   - Every pointer argument is a DEVICE pointer owned by the caller, except
 *     `pool` (a host pointer to a small descriptor read during the call).
 *   - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream).  The library allocates no memory per call.
 *   - Host-detectable errors (NULL pointers, unsupported shapes, misaligned
 *     pointers, workspace too small) are returned before anything is
 *     enqueued.  Errors found in the data on the device (a block id outside
 *     the pool, a slot outside the pool, a context length of 0 or beyond the
 *     block table, inconsistent chunk metadata) are recorded in a per-device
 *     error word, the offending row or page is skipped, and nothing traps;
 *     read and clear the word with pa_get_device_error().
 *   - head_dim is 128 and block_size is 16.  q, the pool and out share one
 *     dtype (fp16 or bf16).  Accumulation is fp32.
 *   - Kernels are launched with programmatic dependent launch: each may start
 *     while the kernel enqueued just before it on `stream` is finishing, and
 *     waits for that kernel to complete before it reads the pool, q or k/v.
 *     The attention calls read block_tables, context_lens and the chunk
 *     metadata BEFORE that wait.  A caller kernel enqueued right before them
 *     that signals programmatic launch completion early
 *     (griddepcontrol.launch_dependents / cudaTriggerProgrammaticLaunchCompletion)
 *     must therefore not write those arrays after its signal.  Kernels that
 *     never signal (every PyTorch kernel, for one) are safe: the attention
 *     kernel then starts only once they have ended.
 *   - Per-context state: the device addresses of the library's own device
 *     variables (the error word, the allocation-free decode's scratch) are
 *     looked up once per CUDA context and keyed on its unique id, so calls
 *     from a driver-API context of the host application, or after
 *     cudaDeviceReset(), look them up anew in that context.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 10
#define PA_HEAD_DIM 128
#define PA_BLOCK_SIZE 16
#define PA_MAX_CHUNK_LEN 512 /* [P1] scheduler task 12.4: prefill chunks of at most 512 tokens */

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef void *pa_stream_t; /* a cudaStream_t */

typedef enum { PA_F16 = 0, PA_BF16 = 1 } pa_dtype;

typedef enum {
  PA_OK = 0,
  PA_ERR_NULL = -1,        /* a required pointer is NULL */
  PA_ERR_SHAPE = -2,       /* a size is negative, inconsistent or over a limit */
  PA_ERR_DTYPE = -3,       /* dtype is neither PA_F16 nor PA_BF16 */
  PA_ERR_UNSUPPORTED = -4, /* head_dim != 128, block_size != 16, or an unsupported head ratio */
  PA_ERR_WORKSPACE = -5,   /* workspace missing or smaller than the size query returns */
  PA_ERR_CUDA = -6,        /* a CUDA runtime/driver call failed (see pa_last_cuda_error) */
  PA_ERR_RANGE = -7,       /* device: block id / slot / context length out of range */
  PA_ERR_TIMEOUT = -8,     /* device: a bounded wait on an asynchronous copy gave up */
  PA_ERR_ALIGN = -9,       /* a pointer is not 16-byte aligned */
  PA_ERR_NO_BLOCKS = -10,  /* allocator: not enough free blocks (nothing was allocated) */
  PA_ERR_STATE = -11       /* allocator: a call out of order (release of a free block, commit beyond
                              the reservation, adopt or fork into a non-empty sequence, ...) */
} pa_status;

/*
 * One layer's KV pool [P1, qwen_serve/paged.py, PagedKVCache docstring]:
 * k_cache and v_cache are each [num_blocks][block_size][num_kv_heads][head_dim]
 * contiguous; block b is the outer index, the in-block slot the next one.
 * The flat slot of (block b, offset o) is b * block_size + o.
 */
typedef struct {
  void *k_cache;
  void *v_cache;
  int32_t num_blocks;
  int32_t block_size;   /* must be 16 */
  int32_t num_kv_heads;
  int32_t head_dim;     /* must be 128 */
  int32_t dtype;        /* pa_dtype */
} pa_kv_pool;

/*
 * kv_cache_write — [P1, qwen_serve/paged.py, PagedKVCache.write]: copy the
 * K and V rows of num_tokens new tokens into their slots.
 *   k, v          [num_tokens][num_kv_heads][128], pool dtype.
 *   slot_mapping  int64 [num_tokens]: flat slot (block * 16 + offset) of each
 *                 token, composed by the caller from its block table as
 *                 table[pos / 16] * 16 + pos % 16.
 * A bit copy: the pool afterwards holds exactly the input bits.  A slot outside
 * [0, num_blocks * 16) records PA_ERR_RANGE and that token is skipped.  Two
 * tokens with the same slot in one call race (undefined which one lands).
 * num_tokens == 0 is a no-op.
 */
PA_API pa_status pa_kv_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                            int32_t num_tokens, const pa_kv_pool *pool, pa_stream_t stream);

/*
 * Size in bytes of the scratch workspace pa_paged_attn_decode needs for up to
 * num_seqs sequences (split-K partial results plus a small index).  Depends
 * only on its arguments; returns 0 for invalid arguments.
 */
PA_API size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t max_context_len);

/*
 * paged_attn_decode — [P1, qwen_serve/model.py, Qwen3Model.forward with one
 * new token per sequence; P2 section 1]: for each sequence s and query head g,
 *   out[s][g] = softmax_j(scale * q[s][g] . K_j) V_j  over j < context_lens[s],
 * where K_j, V_j are KV head g / (num_q_heads / num_kv_heads) of logical
 * position j, read from block block_tables[s][j / 16] at in-block offset j % 16.
 * The new token's K/V must already be in the pool (write first), so
 * context_lens[s] counts it.
 *   q             [num_seqs][num_q_heads][128], pool dtype.
 *   block_tables  int32 [num_seqs][max_blocks_per_seq]; entries past
 *                 ceil(context_lens[s] / 16) are never read.
 *   context_lens  int32 [num_seqs], each in [1, max_blocks_per_seq * 16].
 *   max_context_len  host-side upper bound on context_lens (sizes the launch
 *                 and the workspace; a larger length is still computed).
 *   out           [num_seqs][num_q_heads][128], pool dtype.
 *   workspace     at least pa_decode_workspace_bytes(num_seqs, num_q_heads,
 *                 num_kv_heads, max_context_len) bytes, 16-byte aligned; its
 *                 contents need no initialisation and are clobbered.
 * num_q_heads / num_kv_heads must be 1, 2, 4 or 8.  A sequence whose length is
 * 0 or beyond its table records PA_ERR_RANGE; its output rows are untouched.
 */
PA_API pa_status pa_paged_attn_decode(const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *context_lens,
                               int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                               float scale, void *out, void *workspace, size_t workspace_bytes,
                               pa_stream_t stream);

/*
 * paged_attn_decode_append — the KV write of each sequence's new token fused
 * into the decode: equivalent to pa_kv_cache_write of k_new[s], v_new[s] into
 * slot block_tables[s][(context_lens[s] - 1) / 16] * 16 + (context_lens[s] - 1) % 16
 * (the position after the cached ones, [P1 PagedKVCache.write]) followed by
 * pa_paged_attn_decode, in one launch (or two on the split path): the warp
 * that streams a sequence's last page writes the new row into the pool and
 * into its copy of that page.  16-bit pools only.
 *   k_new, v_new  [num_seqs][num_kv_heads][128], pool dtype, 16-byte aligned.
 * Other arguments, workspace and errors as pa_paged_attn_decode; a sequence
 * whose length is out of range writes nothing.
 */
PA_API pa_status pa_paged_attn_decode_append(const void *q, const void *k_new, const void *v_new,
                                             const pa_kv_pool *pool, const int32_t *block_tables,
                                             int32_t max_blocks_per_seq, const int32_t *context_lens,
                                             int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                                             float scale, void *out, void *workspace, size_t workspace_bytes,
                                             pa_stream_t stream);

/*
 * paged_attn_decode_ex — one decode call with every option:
 *   window        sliding window in keys as pa_paged_attn_decode_window (0: none);
 *   k_new, v_new  the fused KV write of pa_paged_attn_decode_append (both NULL:
 *                 none; not combined with a window: PA_ERR_UNSUPPORTED);
 *   flags         0, or PA_DECODE_EARLY_PAGES: a promise by the caller that the
 *                 work enqueued on `stream` just before this call writes no
 *                 pool page this call reads other than each sequence's last
 *                 visible page (the page of position context_lens[s] - 1), as
 *                 in a decode step whose KV write adds one token per sequence.
 *                 When that work is a pa_kv_cache_write, which lets the next
 *                 kernel start beside the tail of the work before it, the
 *                 promise covers that earlier work too.  The one-launch path
 *                 then starts fetching the other pages before that work has
 *                 finished, overlapping it (the results do not change).
 *                 Breaking the promise gives undefined results.
 *                 PA_DECODE_ZEROED_WORKSPACE: a promise that the workspace
 *                 was zero-filled before its first use and has since been
 *                 used only by calls that completed without PA_ERR_TIMEOUT
 *                 (every such call leaves the workspace's item counters at
 *                 zero again).  The call then runs as ONE kernel over all
 *                 SMs whatever the sizes: pages are dealt evenly to every
 *                 warp the GPU holds, and the warp that finishes the last
 *                 piece of a split (sequence, KV head) merges the pieces
 *                 (log-sum-exp) from L2, counting arrivals in the workspace.
 *                 After a PA_ERR_TIMEOUT, zero-fill the workspace again.
 *                 Other bits: PA_ERR_UNSUPPORTED.
 * Other arguments, workspace and errors as pa_paged_attn_decode.  No
 * counterpart on the pages: a library addition.
 */
#define PA_DECODE_EARLY_PAGES 1u
#define PA_DECODE_ZEROED_WORKSPACE 2u
PA_API pa_status pa_paged_attn_decode_ex(const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                                         int32_t max_blocks_per_seq, const int32_t *context_lens,
                                         int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                                         float scale, int32_t window, const void *k_new, const void *v_new,
                                         uint32_t flags, void *out, void *workspace, size_t workspace_bytes,
                                         pa_stream_t stream);

/*
 * Number of kernels one pa_paged_attn_decode (or _noalloc) call with these
 * arguments launches on the current device: 1 when every (sequence, KV head)
 * pair gets its own SMs and a pair of max_context_len tokens, streamed by
 * them, would still end before a split launch over the whole GPU (the pair
 * merges its warps' partial results on chip); 2 (split-K pass, then the
 * combine pass) otherwise.  With 8 KV heads on 152 SMs: up to 9 sequences of
 * up to 3072 tokens, or up to 19 of up to 1488 tokens, take one launch.  The
 * choice depends only on these arguments and the device's SM count.
 * Returns 0 for arguments the call would reject or with no work (num_seqs 0).
 */
PA_API int32_t pa_decode_kernel_launches(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len);

/*
 * paged_attn_decode_noalloc — no counterpart on the pages: a library addition
 * for callers that cannot allocate device memory or pass a workspace (a
 * plugin inside a host application that owns all device memory, a serving
 * step that must not allocate).  Same arguments and result as
 * pa_paged_attn_decode without the workspace: the split-K scratch is one
 * fixed array of PA_NOALLOC_SCRATCH_BYTES inside the library, held by every
 * GPU that loads the library until the process exits.  A call whose
 * pa_decode_workspace_bytes(...) exceeds PA_NOALLOC_SCRATCH_BYTES returns
 * PA_ERR_WORKSPACE and enqueues nothing (with 8 KV heads this admits head
 * ratios up to 4: e.g. up to ~7900 (sequence, KV head) pairs at ratio 4; a
 * ratio of 8 never fits).  Argument errors are checked first, in the order
 * pa_paged_attn_decode checks them, so a call that is both malformed and too
 * large returns the argument error.  It calls no allocator.  The first call in
 * a CUDA context (with that context's device current) looks up the array's
 * device address; make it before any stream capture.  All calls share the
 * array, which keeps the last call's contents (nothing in it needs to start at
 * zero); calls that overlap on the GPU race on it, so serialise them.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)
PA_API pa_status pa_paged_attn_decode_noalloc(const void *q, const pa_kv_pool *pool,
                                              const int32_t *block_tables, int32_t max_blocks_per_seq,
                                              const int32_t *context_lens, int32_t num_seqs,
                                              int32_t num_q_heads, int32_t max_context_len, float scale,
                                              void *out, pa_stream_t stream);

/*
 * paged_attn_prefill_chunk — [P1, qwen_serve/model.py, Qwen3Model.forward
 * with T > 1: causal mask kpos <= qpos on absolute positions; P2 section 3.4
 * and task 04.1]: chunk c has chunk_lens[c] new query tokens at absolute
 * positions chunk_starts[c] + i, attending to keys 0 .. chunk_starts[c] + i
 * of its own sequence, read through block_tables[c].
 *   q             [total_q_tokens][num_q_heads][128]: the chunks' rows packed
 *                 in chunk order (chunk c starts at row sum_{c'<c} chunk_lens[c']).
 *   chunk_starts, chunk_lens, context_lens  int32 [num_chunks];
 *                 context_lens[c] must equal chunk_starts[c] + chunk_lens[c]
 *                 (the chunk's own K/V are written first), and
 *                 1 <= chunk_lens[c] <= max_chunk_len.
 *   block_tables  int32 [num_chunks][max_blocks_per_seq].
 *   max_chunk_len host-side bound on chunk_lens, at most 512.
 *   out           [total_q_tokens][num_q_heads][128], pool dtype.
 * QK^T and PV run on the tensor cores (bf16 or fp16 operands, fp32
 * accumulation); the probabilities enter PV rounded to the input dtype.
 * num_q_heads / num_kv_heads must be 1, 2, 4 or 8.  A chunk with inconsistent
 * metadata records PA_ERR_RANGE and its rows are untouched.
 */
PA_API pa_status pa_paged_attn_prefill_chunk(const void *q, const int32_t *chunk_starts,
                                      const int32_t *chunk_lens, const pa_kv_pool *pool,
                                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                                      const int32_t *context_lens, int32_t num_chunks,
                                      int32_t num_q_heads, int32_t total_q_tokens,
                                      int32_t max_chunk_len, float scale, void *out,
                                      pa_stream_t stream);

/*
 * ---- int8 KV pool [P2 section 5, KV8Cache] ----------------------------------
 * One layer's pool with int8 codes instead of 16-bit values: K and V codes
 * [num_blocks][16][num_kv_heads][128] (the same slot addressing), and one fp32
 * scale per (token, KV head) for K and one for V, stored
 * [num_blocks][num_kv_heads][16] (head-major inside a block, so the 16 scales
 * of one page of one KV head are 64 contiguous bytes).  Half the bytes of a
 * 16-bit pool plus 8 bytes per token and KV head.  All four arrays are
 * caller-owned device memory, 16-byte aligned.
 */
typedef struct {
  void *k_cache;        /* int8 codes */
  void *v_cache;
  float *k_scale;       /* fp32 scales */
  float *v_scale;
  int32_t num_blocks;
  int32_t block_size;   /* must be 16 */
  int32_t num_kv_heads;
  int32_t head_dim;     /* must be 128 */
} pa_kv_pool_q8;

/*
 * kv_cache_write_q8 — [P2 section 5, KV8Cache.write]: quantise the K and V
 * rows of num_tokens new tokens into their slots of an int8 pool.  For each
 * token and KV head, separately for K and V: scale = max |x| / 127 + 1e-8 and
 * code = clip(rint(x / scale), -127, 127), in fp32 with every operation
 * rounded to nearest (ties to even), so codes and scales are bit-exact.
 *   k, v          [num_tokens][num_kv_heads][128] in `dtype` (PA_F16 / PA_BF16).
 *   slot_mapping  int64 [num_tokens] as for pa_kv_cache_write; a slot outside
 *                 the pool records PA_ERR_RANGE and is skipped.
 */
PA_API pa_status pa_kv_cache_write_q8(const void *k, const void *v, int32_t dtype, const int64_t *slot_mapping,
                                      int32_t num_tokens, const pa_kv_pool_q8 *pool, pa_stream_t stream);

/*
 * paged_attn_decode_q8 — pa_paged_attn_decode over an int8 pool: keys and
 * values are the dequantised numbers code * scale [P2 section 5,
 * KV8Cache.read]; q and out are `dtype` (PA_F16 / PA_BF16).  Arguments,
 * workspace (pa_decode_workspace_bytes) and errors as pa_paged_attn_decode.
 */
PA_API pa_status pa_paged_attn_decode_q8(const void *q, int32_t dtype, const pa_kv_pool_q8 *pool,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_context_len, float scale, void *out, void *workspace,
                                         size_t workspace_bytes, pa_stream_t stream);

/*
 * ---- fp8 KV pool [P2 sections 5.1 and 5.4 (FP8 storage of K and V)] --------
 * The pa_kv_pool_q8 layout and scales with FP8 E4M3 codes (the "fn" format:
 * bias 7, 3 fraction bits, largest finite 448, no infinity) in k_cache and
 * v_cache instead of int8 integers.
 *
 * kv_cache_write_f8 — as pa_kv_cache_write_q8 with scale = max |x| / 448 +
 * 1e-8 and code = the E4M3 value nearest to the fp32 quotient x / scale (ties
 * to even; the quotient never exceeds 448 in magnitude), so codes and scales
 * are bit-exact.  Same arguments and errors.
 */
PA_API pa_status pa_kv_cache_write_f8(const void *k, const void *v, int32_t dtype, const int64_t *slot_mapping,
                                      int32_t num_tokens, const pa_kv_pool_q8 *pool, pa_stream_t stream);

/*
 * paged_attn_decode_f8 — pa_paged_attn_decode over an fp8 pool: keys and
 * values are the dequantised numbers e4m3(code) * scale.  Arguments, workspace
 * (pa_decode_workspace_bytes) and errors as pa_paged_attn_decode_q8.
 */
PA_API pa_status pa_paged_attn_decode_f8(const void *q, int32_t dtype, const pa_kv_pool_q8 *pool,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_context_len, float scale, void *out, void *workspace,
                                         size_t workspace_bytes, pa_stream_t stream);

/*
 * paged_attn_decode_q8_ex — the decode over an 8-bit pool with flags:
 *   codes   PA_CODES_INT8 (as pa_paged_attn_decode_q8) or PA_CODES_E4M3 (as
 *           pa_paged_attn_decode_f8); anything else: PA_ERR_UNSUPPORTED;
 *   flags   PA_DECODE_EARLY_PAGES and PA_DECODE_ZEROED_WORKSPACE, with the
 *           promises stated at pa_paged_attn_decode_ex (pa_kv_cache_write_q8
 *           / _f8 let the next kernel start beside the tail of the work before
 *           them, as pa_kv_cache_write does); other bits: PA_ERR_UNSUPPORTED.
 * Other arguments, workspace and errors as pa_paged_attn_decode_q8.  No
 * counterpart on the pages: a library addition.
 */
#define PA_CODES_INT8 0
#define PA_CODES_E4M3 1
PA_API pa_status pa_paged_attn_decode_q8_ex(const void *q, int32_t dtype, const pa_kv_pool_q8 *pool, int32_t codes,
                                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                                            const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                            int32_t max_context_len, float scale, uint32_t flags, void *out,
                                            void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * paged_attn_prefill_chunk_q8 — [P2 section 5 (KV8Cache: one int8 cache read
 * by every attention call) and section 5.4 (FP8 KV)]: the causal chunked
 * prefill of pa_paged_attn_prefill_chunk over an 8-bit pool; every key and
 * value is the dequantised number code * scale.
 *   q, out      [total_q_tokens][num_q_heads][128] of `dtype` (PA_F16 or
 *               PA_BF16; the pool's codes carry no dtype); else PA_ERR_DTYPE.
 *   codes       PA_CODES_INT8 or PA_CODES_E4M3 (the codes written by
 *               pa_kv_cache_write_q8 / _f8); else PA_ERR_UNSUPPORTED.
 * Other arguments, and errors, as pa_paged_attn_prefill_chunk (chunk metadata
 * and block ids checked on the device; a bad chunk is reported and left
 * unwritten, a page with a block id outside the pool is reported and
 * skipped).  No sliding window.  Runs on the tcgen05 tensor cores with fp16
 * operands: each key and value code * scale is rounded once to fp16 in shared
 * memory; a bf16 query is exact in fp16 after scaling each row by a power of
 * two (an fp16 query is used as is); scores and sums fp32, the probabilities
 * rounded to fp16 for the P V product, the output in `dtype`.  A dequantised
 * key or value beyond the fp16 range (65504) saturates to it.
 */
PA_API pa_status pa_paged_attn_prefill_chunk_q8(const void *q, int32_t dtype, const int32_t *chunk_starts,
                                                const int32_t *chunk_lens, const pa_kv_pool_q8 *pool, int32_t codes,
                                                const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                const int32_t *context_lens, int32_t num_chunks,
                                                int32_t num_q_heads, int32_t total_q_tokens, int32_t max_chunk_len,
                                                float scale, void *out, pa_stream_t stream);

/*
 * mixed_step — [P2 section 3.4 (a step that prefills chunks of new prompts
 * while running sequences decode one token each, the chunks reading their
 * cached prefix); P1 "Куда расти" (production engines fuse the step into
 * dedicated kernels)]: a whole mixed step over a 16-bit pool in ONE
 * persistent launch (one CTA per SM, launched cooperatively), its SMs split
 * between the chunks and the sequences by their work:
 *   chunks      the KV write of the chunks' num_chunk_tokens new tokens,
 *               exactly as pa_kv_cache_write (k_chunks, v_chunks
 *               [num_chunk_tokens][Hkv][128] of the pool's dtype, chunk_slots
 *               int64; a bad slot is reported and skipped), then, once every
 *               such row is written (a barrier of the prefill CTAs, bounded:
 *               PA_ERR_TIMEOUT), the chunked prefill of
 *               pa_paged_attn_prefill_chunk (q_chunks, chunk_starts,
 *               chunk_lens, chunk_block_tables [num_chunks][chunk_max_blocks],
 *               chunk_context_lens, total_q_tokens, max_chunk_len, out_chunks;
 *               num_chunks <= 256, no window);
 *   sequences   the decode of pa_paged_attn_decode_append (q, k_dec, v_dec
 *               [num_seqs][Hkv][128]: each sequence's new token, written at
 *               position context_lens[s] - 1 by the decode as it reads that
 *               page; k_dec = v_dec = NULL: the new tokens are already in the
 *               pool; block_tables [num_seqs][max_blocks_per_seq],
 *               context_lens, out; num_seqs <= 6000), which does not wait for
 *               the chunks' write.  So no sequence may read a slot of the
 *               chunks' write, and no chunk may read a page that holds a
 *               sequence's new token (both hold when a scheduler gives the
 *               new tokens of each chunk and sequence pages of their own).
 * Either part may be empty (num_chunks = num_chunk_tokens = 0, or num_seqs =
 * 0; its pointers are then not read).  Results as the separate calls (the
 * chunks' write first).
 *   workspace   pa_mixed_step_workspace_bytes(num_seqs, num_q_heads,
 *               num_kv_heads) bytes, 16-byte aligned, zero-filled before its
 *               first use; every call that completes without PA_ERR_TIMEOUT
 *               leaves its counters zero again, so it needs no clearing
 *               between calls.  After a PA_ERR_TIMEOUT, zero-fill it again.
 *               Missing or too small: PA_ERR_WORKSPACE.
 * Other checks and errors as the separate calls.  No counterpart on the
 * pages: a library addition.
 */
PA_API size_t pa_mixed_step_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads);
PA_API pa_status pa_mixed_step(const pa_kv_pool *pool, int32_t num_q_heads, float scale, const void *k_chunks,
                               const void *v_chunks, const int64_t *chunk_slots, int32_t num_chunk_tokens,
                               const void *q_chunks, const int32_t *chunk_starts, const int32_t *chunk_lens,
                               const int32_t *chunk_block_tables, int32_t chunk_max_blocks,
                               const int32_t *chunk_context_lens, int32_t num_chunks, int32_t total_q_tokens,
                               int32_t max_chunk_len, void *out_chunks, const void *q, const void *k_dec,
                               const void *v_dec, const int32_t *block_tables, int32_t max_blocks_per_seq,
                               const int32_t *context_lens, int32_t num_seqs, void *out, void *workspace,
                               size_t workspace_bytes, pa_stream_t stream);

/*
 * ---- sliding window [P2 section 4 (a ring of capacity W keeps the last W
 * tokens; the mask stays on absolute positions) and section 5.2 (window
 * attention)] -------------------------------------------------------------------
 * With window W >= 1 a query at absolute position p attends only to keys
 * max(0, p - W + 1) .. p; window 0 means no window (the plain calls).  Blocks
 * wholly before a sequence's (or chunk's first query's) window are never read:
 * their block-table entries may already hold -1 or point at reused blocks.
 */

/*
 * paged_attn_decode_window — pa_paged_attn_decode with a sliding window of
 * `window` keys: sequence s attends to j in [max(0, context_lens[s] - window),
 * context_lens[s]).  Arguments, workspace and errors as pa_paged_attn_decode;
 * window < 0 returns PA_ERR_SHAPE.  A sequence's window spans at most
 * (window - 1) / 16 + 2 pages, so the call launches the kernels
 * pa_decode_kernel_launches gives for max_context_len =
 * min(max_context_len, 16 * ((window - 1) / 16 + 2)).
 */
PA_API pa_status pa_paged_attn_decode_window(const void *q, const pa_kv_pool *pool, const int32_t *block_tables,
                                             int32_t max_blocks_per_seq, const int32_t *context_lens,
                                             int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len,
                                             float scale, int32_t window, void *out, void *workspace,
                                             size_t workspace_bytes, pa_stream_t stream);

/*
 * paged_attn_prefill_chunk_window — pa_paged_attn_prefill_chunk with a
 * sliding window of `window` keys: the query at position chunk_starts[c] + i
 * attends to keys max(0, chunk_starts[c] + i - window + 1) ..
 * chunk_starts[c] + i.  Arguments and errors as pa_paged_attn_prefill_chunk;
 * window < 0 returns PA_ERR_SHAPE.
 */
PA_API pa_status pa_paged_attn_prefill_chunk_window(const void *q, const int32_t *chunk_starts,
                                                    const int32_t *chunk_lens, const pa_kv_pool *pool,
                                                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                                                    const int32_t *context_lens, int32_t num_chunks,
                                                    int32_t num_q_heads, int32_t total_q_tokens,
                                                    int32_t max_chunk_len, float scale, int32_t window,
                                                    void *out, pa_stream_t stream);

/*
 * paged_attn_prefill_chunk_ex — pa_paged_attn_prefill_chunk_window (window 0:
 * the plain causal chunks) as one launch balanced over the SMs.  No
 * counterpart on the pages: a library addition.  The causal mask makes a
 * chunk's last query tiles many times heavier than its first ones (and a long
 * prefix heavier still); here one CTA per SM takes an equal share of all
 * (query tile, 128-key tile) pairs, and a query tile split between CTAs is
 * merged (log-sum-exp) by the CTA whose piece finishes last.
 *   workspace  at least pa_prefill_workspace_bytes(...) bytes (for the current
 *              device: it depends on its SM count), 16-byte aligned.  Zero-fill
 *              it before its first use; every call that completes without
 *              PA_ERR_TIMEOUT leaves its counters at zero again, so it needs no
 *              clearing between calls (after a PA_ERR_TIMEOUT, zero-fill it
 *              again).  Calls sharing a workspace must not overlap on the GPU.
 * With more than 256 chunks the plain launch runs (the workspace is unused).
 * Results equal the plain call's up to fp32 rounding (a split tile's pieces
 * are summed in another order).  Other arguments and errors as
 * pa_paged_attn_prefill_chunk_window; no workspace: PA_ERR_WORKSPACE.
 */
PA_API size_t pa_prefill_workspace_bytes(int32_t num_chunks, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t max_chunk_len);
PA_API pa_status pa_paged_attn_prefill_chunk_ex(const void *q, const int32_t *chunk_starts, const int32_t *chunk_lens,
                                                const pa_kv_pool *pool, const int32_t *block_tables,
                                                int32_t max_blocks_per_seq, const int32_t *context_lens,
                                                int32_t num_chunks, int32_t num_q_heads, int32_t total_q_tokens,
                                                int32_t max_chunk_len, float scale, int32_t window, void *out,
                                                void *workspace, size_t workspace_bytes, pa_stream_t stream);

/*
 * qk_norm_rope_kv_write — [P1, qwen_serve/model.py: rms_norm, _rotate_half,
 * apply_rope and Qwen3Model.forward (q_norm / k_norm, then the rotary embedding
 * at each token's absolute position, then PagedKVCache.write); P2 section 4:
 * the key is rotated before it is stored]: for each new token t,
 *   q_out[t][g] = rope(rms_norm(q[t][g], q_norm_weight), positions[t])  (every query head g),
 *   slot_mapping[t] receives K = rope(rms_norm(k[t][h], k_norm_weight), positions[t]) and V = v[t][h].
 * rms_norm(x, w) = round(round(x * inv) * w), inv = rsqrt(mean(x^2) + eps) in
 * fp32 (the fp32 mean nearest the exact one, a correctly rounded reciprocal
 * square root); rope(z) = round(round(z * cos) + round(rotate_half(z) * sin))
 * with rotate_half(z) = (-z[64..128), z[0..64)) (NeoX layout), the tables'
 * row positions[t]; round() is to the pool dtype, ties to even, and every
 * product and sum is exact in fp32 before it.  The result is bit-exact.
 *   q, q_out      [num_tokens][num_q_heads][128], pool dtype; q_out may be q.
 *   k, v          [num_tokens][num_kv_heads][128], pool dtype.
 *   q_norm_weight, k_norm_weight  [128], pool dtype.
 *   cos_table, sin_table  [max_position][128], pool dtype (the caller's
 *                 rotary tables, e.g. theta^(-2i/128) frequencies, halves duplicated).
 *   positions     int32 [num_tokens] absolute positions; slot_mapping int64
 *                 [num_tokens] as for pa_kv_cache_write.
 * A token whose position lies outside [0, max_position) or whose slot lies
 * outside the pool records PA_ERR_RANGE (detail: the token) and nothing of it
 * is written.  All pointers 16-byte aligned (positions 4, slot_mapping 8).
 */
PA_API pa_status pa_qk_norm_rope_kv_write(const void *q, const void *k, const void *v, const void *q_norm_weight,
                                          const void *k_norm_weight, float eps, const void *cos_table,
                                          const void *sin_table, int32_t max_position, const int32_t *positions,
                                          const int64_t *slot_mapping, int32_t num_tokens, int32_t num_q_heads,
                                          void *q_out, const pa_kv_pool *pool, pa_stream_t stream);

/*
 * ---- copy-on-write and the block-table builder [P1, qwen_serve/paged.py:
 * BlockAllocator, SequenceCache.fork_from / _cow_copy / adopt_prefix /
 * reserve / commit; task 12.1 worked examples and acceptance item 5] --------
 */

/*
 * kv_block_copy — [P1, SequenceCache._cow_copy: k[:, dst] = k[:, src] and the
 * same for v, over every layer]: for each pair i and each of num_layers
 * pools, copy physical block pairs[2i] (src) onto block pairs[2i + 1] (dst)
 * in both k_cache and v_cache.  A bit copy.
 *   pools      HOST array [num_layers] of layer pools with one geometry
 *              (num_blocks, num_kv_heads, dtype); read during the call.
 *   pairs      DEVICE int32 [num_pairs][2] (src, dst).  The dst blocks must
 *              be distinct and none may be a src of the same call (as with
 *              blocks fresh from the allocator); otherwise the result is
 *              undefined.  src == dst is a no-op.
 * A pair with a block outside [0, num_blocks) records PA_ERR_RANGE (detail:
 * the pair index) and is skipped.  num_pairs == 0 is a no-op.
 */
PA_API pa_status pa_kv_block_copy(const pa_kv_pool *pools, int32_t num_layers, const int32_t *pairs,
                                  int32_t num_pairs, pa_stream_t stream);

/*
 * Host-side block allocator and per-sequence block tables (pure host code:
 * none of these calls touches the GPU; not thread-safe — one thread per
 * allocator and its sequences).
 *
 * pa_allocator: a pool of num_blocks block ids with a reference count each;
 * free ids are handed out first-in first-out (ids 0, 1, 2, ... on a new
 * allocator) and a released id goes to the back of the free list.
 * pa_sequence: one request's block table and committed length.  reserve()
 * makes room for the next tokens and returns their flat slots; the caller
 * writes their K/V (pa_kv_cache_write) and then commit()s them.  fork()
 * shares every block of another sequence by reference (+1 each); the first
 * reserve() that writes into a shared, partly filled block replaces it with a
 * fresh copy (copy-on-write): the allocator records the (src, dst) pair,
 * which the caller takes with pa_allocator_take_copies() and enqueues with
 * pa_kv_block_copy() before that step's KV write.
 */
typedef struct pa_allocator pa_allocator;
typedef struct pa_sequence pa_sequence;

typedef struct {
  int32_t total;         /* num_blocks */
  int32_t free;          /* ids in the free list */
  int32_t used;          /* ids with refcount > 0 (used + free == total) */
  int32_t shared;        /* ids with refcount > 1 */
  int64_t n_allocated;   /* ids handed out so far */
  int64_t n_cow;         /* copy-on-write events so far */
} pa_allocator_stats;

/* A new allocator of num_blocks (>= 1) ids, all free; *out receives it. */
PA_API pa_status pa_allocator_create(int32_t num_blocks, pa_allocator **out);
/* Frees the allocator (its sequences must be destroyed first). */
PA_API void pa_allocator_destroy(pa_allocator *alloc);
/* n ids with refcount 1 into out[0..n); all or nothing: PA_ERR_NO_BLOCKS if
 * fewer than n are free (the pages' OutOfBlocks). */
PA_API pa_status pa_allocator_allocate(pa_allocator *alloc, int32_t n, int32_t *out);
/* +1 on an id in use; PA_ERR_STATE on a free id, PA_ERR_RANGE outside the pool. */
PA_API pa_status pa_allocator_retain(pa_allocator *alloc, int32_t block);
/* -1; at 0 the id returns to the back of the free list.  PA_ERR_STATE on a free id. */
PA_API pa_status pa_allocator_release(pa_allocator *alloc, int32_t block);
/* Reference count of an id (-1 outside the pool). */
PA_API int32_t pa_allocator_refcount(const pa_allocator *alloc, int32_t block);
PA_API pa_status pa_allocator_stats_get(const pa_allocator *alloc, pa_allocator_stats *out);
/* Moves the recorded copy-on-write pairs (src, dst) into pairs[0 .. 2 *num):
 * *num receives their count.  If capacity (in pairs) is too small, nothing
 * is moved, *num receives the count needed and PA_ERR_SHAPE is returned. */
PA_API pa_status pa_allocator_take_copies(pa_allocator *alloc, int32_t *pairs, int32_t capacity, int32_t *num);

/* A new, empty sequence on `alloc`; *out receives it. */
PA_API pa_status pa_sequence_create(pa_allocator *alloc, pa_sequence **out);
/* Releases the sequence's blocks and frees it. */
PA_API void pa_sequence_destroy(pa_sequence *seq);
/* Room for n more tokens after the committed and already reserved ones:
 * allocates the blocks they need (and the copy of a shared partly filled
 * block they would write into); writes the n flat slots (block * 16 +
 * offset) into slots (may be NULL).  All or nothing (PA_ERR_NO_BLOCKS). */
PA_API pa_status pa_sequence_reserve(pa_sequence *seq, int32_t n, int64_t *slots);
/* Marks the first n reserved tokens as written (n <= reserved, else PA_ERR_STATE). */
PA_API pa_status pa_sequence_commit(pa_sequence *seq, int32_t n);
/* Starts an empty sequence on n full blocks in use elsewhere (a shared
 * prefix): each gains a reference; length = 16 n.  PA_ERR_STATE if the
 * sequence is not empty or a block is free. */
PA_API pa_status pa_sequence_adopt_prefix(pa_sequence *seq, const int32_t *blocks, int32_t n);
/* Makes the empty sequence `seq` a copy of `other` (same allocator, nothing
 * reserved): every block is shared by reference, the length is copied. */
PA_API pa_status pa_sequence_fork(pa_sequence *seq, const pa_sequence *other);
/* Releases every block; the sequence is empty again. */
PA_API pa_status pa_sequence_release(pa_sequence *seq);
/* Committed tokens, reserved-but-uncommitted tokens, and blocks held. */
PA_API int32_t pa_sequence_length(const pa_sequence *seq);
PA_API int32_t pa_sequence_reserved(const pa_sequence *seq);
PA_API int32_t pa_sequence_num_blocks(const pa_sequence *seq);
/* Copies the block ids into out[0 .. num_blocks) (capacity must suffice). */
PA_API pa_status pa_sequence_blocks(const pa_sequence *seq, int32_t *out, int32_t capacity);
/*
 * The step's metadata for the attention calls, into HOST arrays: for
 * sequence i, block_tables[i][0 .. max_blocks) = its block ids padded with -1,
 * chunk_starts[i] = committed length, chunk_lens[i] = reserved tokens and
 * context_lens[i] = their sum (a decode sequence reserves 1).  Any of the
 * last three may be NULL.  PA_ERR_SHAPE if a sequence holds more than
 * max_blocks blocks.
 */
PA_API pa_status pa_build_step_tables(const pa_sequence *const *seqs, int32_t num_seqs, int32_t max_blocks,
                                      int32_t *block_tables, int32_t *chunk_starts, int32_t *chunk_lens,
                                      int32_t *context_lens);

/*
 * Synchronises `stream`, then returns and clears the current device's error
 * word (PA_OK if no kernel recorded an error).  If `detail` is not NULL it
 * receives the index (token, sequence or chunk) of the first error.
 */
PA_API pa_status pa_get_device_error(pa_stream_t stream, int32_t *detail);

/*
 * Self-test of failure detection: launches one warp that waits, with the
 * same bounded wait every kernel of the library uses on its copies and MMAs,
 * on a barrier that nothing completes.  After limit_us microseconds (1 ..
 * 2,000,000) the wait gives up, PA_ERR_TIMEOUT (detail -1) is recorded in the
 * device error word and the kernel returns: pa_get_device_error() then
 * reports it and the context stays usable.  Nothing faults, traps or hangs.
 */
PA_API pa_status pa_selftest_bounded_wait(uint32_t limit_us, pa_stream_t stream);

/* Human-readable name of a status code (static storage). */
PA_API const char *pa_status_string(int32_t status);

/* The last CUDA error code the library saw on this thread (0 if none). */
PA_API int32_t pa_last_cuda_error(void);

/* PA_ABI_VERSION of the loaded library. */
PA_API int32_t pa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
