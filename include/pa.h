/*
 * pa.h -- C ABI of the paged varlen attention library (libpa.so), sm_103a.
 *
 * The operations follow the web pages that describe vLLM's attention
 * backends:
 *   [FA-vLLM] "FlashAttention 在 vLLM 中的实现分析" (blog.chen3feng.top,
 *             vllm-analysis/07): §1.1 tiled online softmax, §4 forward() and the
 *             flash_attn_varlen_func call, §4.2 KV-cache update, §5 PagedAttention
 *             integration (block_table addressing), §6.3 cascade execution,
 *             §8.2 reshape_and_cache_flash / merge_attn_states, §9 DCP, §10 feature
 *             table.
 *   [FA/FI]   "FlashAttention と FlashInfer:2 大 GPU アテンションバックエンド":
 *             データフロー (KV cache shape, block size multiple of 16),
 *             境界と失敗 (head-size and dtype limits, FP8 KV cache).
 *   [Backend] "AttentionBackend:アテンションバックエンド抽象レイヤー": 境界と失敗
 *             (head size, block size ValueError, natural-log LSE).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library
 *     never allocates device memory: temporaries live in a caller-provided
 *     workspace whose size the *_workspace_size functions return.
 *   - Work is enqueued on the caller's stream (`stream` is a cudaStream_t; NULL
 *     means the legacy default stream). Calls are asynchronous, make no
 *     host<->device copies, never synchronize, and keep no state between calls,
 *     so they can be recorded into a CUDA graph and called from several host
 *     threads on different streams with different workspaces.
 *   - Element type (the dtype argument): PA_BF16 (bfloat16) or PA_F16 (IEEE
 *     half) for Q, K, V and outputs, the same type for all of them within a
 *     call ([FA-vLLM] §2.1 lists float16 and bfloat16 as the supported
 *     dtypes); LSE is float32. The FP8 entry points (pa_*_fp8kv,
 *     pa_reshape_and_cache_fp8, or the fp8 option of pa_*_fwd_ex) hold K and
 *     V in the page pools as e4m3 bytes instead (Q, the new tokens and the
 *     outputs keep dtype). Arithmetic accumulates in float32; P enters the
 *     P V product in dtype (f16 over e4m3 pools).
 *   - Strides are in ELEMENTS. Every tensor pointer must be 16-byte aligned and
 *     every stride a multiple of 8 elements (16 bytes).
 *   - Return value: PA_OK, or an error code. On any host-side error nothing is
 *     launched and nothing is written. PA_ERR_CUDA reports a failed launch.
 *   - dev_status (nullable): a device int32 the kernels OR error bits into
 *     (PA_DEV_*) when they meet metadata they cannot use (a page id outside the
 *     pool, a slot outside the pool, a sequence longer than its page-table row,
 *     a bounded wait that gave up). The offending access is skipped, never
 *     performed: bad metadata cannot make a kernel read or write out of bounds.
 *     The caller clears the word; the library only ORs bits into it.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int pa_status;

#define PA_OK 0
#define PA_ERR_INVALID_ARG 1 /* null pointer, negative size, bad stride/alignment, H % H_kv != 0 */
#define PA_ERR_BLOCK_SIZE 2  /* block_size not a positive multiple of 16, or > 1024 */
#define PA_ERR_UNSUPPORTED 3 /* head_size or dtype not supported (see each entry point) */
#define PA_ERR_WORKSPACE 4   /* workspace NULL, misaligned or smaller than required */
#define PA_ERR_CUDA 5        /* a kernel launch or a CUDA runtime query failed */
#define PA_ERR_NOALLOC_LIMIT 6 /* problem needs more scratch than pa_varlen_fwd_noalloc's fixed buffer */

/* bits OR-ed into *dev_status by the kernels */
#define PA_DEV_BAD_PAGE 1    /* a block_table entry outside [0, num_blocks): its keys read as 0 */
#define PA_DEV_BAD_SLOT 2    /* a slot_mapping entry >= num_blocks * block_size: token skipped */
#define PA_DEV_BAD_SEQLEN 4  /* cu_seqlens_q / seqused_k inconsistent with the stated bounds */
#define PA_DEV_TIMEOUT 8     /* a bounded wait on a pipeline barrier gave up */
#define PA_DEV_CASCADE 16    /* cascade precondition violated (see pa_cascade_fwd) */

#define PA_BF16 0 /* bfloat16 */
#define PA_F16 1  /* IEEE half (float16) */

/* Human-readable name of a pa_status value (static string). */
const char* pa_status_string(pa_status status);

/* ABI version of this header (increments on any signature change). */
int pa_abi_version(void);

/*
 * pa_reshape_and_cache -- the slot_mapping scatter that writes new K/V rows
 * into their pages before attention ([FA-vLLM] §4.2 and §8.2
 * reshape_and_cache_flash; [FA/FI] 役割: the cache write is its own op).
 *
 *   key[t], value[t]  : [num_kv_heads, head_size] rows, token t at
 *                       key + t * key_token_stride (likewise value).
 *   key_cache, value_cache : page pools; page b starts at b * cache_block_stride
 *                       and holds [block_size, num_kv_heads, head_size]
 *                       contiguous (the NHD layout of [FA-vLLM] §5). Passing
 *                       cache_block_stride = 2*block_size*H_kv*D with value_cache
 *                       = key_cache + block_size*H_kv*D addresses a combined
 *                       [num_blocks, 2, block_size, H_kv, D] tensor ([FA/FI]
 *                       データフロー); the [2, num_blocks, ...] layout is two
 *                       plain pools.
 *   slot_mapping[t]   : int64 flat slot; the token goes to page slot / block_size,
 *                       row slot % block_size. slot < 0 skips the token (padding).
 *                       Slots must be distinct (duplicates: unspecified winner).
 * Bit-exact copy; no arithmetic on values.
 */
pa_status pa_reshape_and_cache(const void* key, const void* value, int64_t key_token_stride,
                               int64_t value_token_stride, void* key_cache, void* value_cache,
                               int64_t cache_block_stride, const int64_t* slot_mapping,
                               int num_tokens, int num_kv_heads, int head_size, int block_size,
                               int num_blocks, int dtype, int32_t* dev_status, void* stream);

/*
 * Workspace bytes pa_varlen_fwd needs for these bounds. sm_count is the
 * multiprocessor count of the device the call will run on (0: query the
 * current device). Returns 0 if the arguments are invalid.
 */
size_t pa_varlen_fwd_workspace_size(int num_seqs, int total_q, int max_seqlen_q, int max_seqlen_k,
                                    int num_heads, int num_kv_heads, int head_size, int block_size,
                                    int sm_count);

/*
 * pa_varlen_fwd -- varlen attention over a paged KV cache ([FA-vLLM] §4 call
 * flash_attn_varlen_func(q, k_cache, v_cache, cu_seqlens_q, seqused_k,
 * block_table, ...), §5 addressing, §1.1 tiled online softmax).
 *
 *   q            : [total_q, num_heads, head_size]; token t at q + t*q_token_stride,
 *                  heads contiguous.
 *   key_cache, value_cache, cache_block_stride : as in pa_reshape_and_cache.
 *   cu_seqlens_q : int32 [num_seqs + 1], nondecreasing prefix sums of query
 *                  lengths, cu_seqlens_q[0] = 0, cu_seqlens_q[num_seqs] = total_q.
 *   seqused_k    : int32 [num_seqs], number of keys of each sequence (>= 0).
 *   block_table  : int32 [num_seqs, bt_stride]; logical key j of sequence s is
 *                  row j % block_size of page block_table[s * bt_stride + j / block_size].
 *                  Only entries j / block_size < ceil(seqused_k[s] / block_size)
 *                  are read.
 *   max_seqlen_q, max_seqlen_k : host upper bounds of the query / key lengths
 *                  (used to size launches and the workspace; no device value is
 *                  read on the host). A looser bound gives the same results;
 *                  a sequence above it sets PA_DEV_BAD_SEQLEN.
 *   softmax_scale: multiplies q.k (commonly 1/sqrt(head_size)); any finite
 *                  value (PA_ERR_INVALID_ARG for NaN or infinity). A zero or
 *                  negative scale runs every segment on the split-KV kernel.
 *   causal       : 0 or 1. Causal masking is bottom-right aligned: query i of a
 *                  sequence with q_len queries and kv_len keys sees keys
 *                  j <= kv_len - q_len + i (a decode query sees all keys).
 *   GQA          : query head h reads KV head h / (num_heads / num_kv_heads);
 *                  any ratio (num_heads % num_kv_heads == 0). Groups of more
 *                  than 128 heads run every segment on the split-KV kernel.
 *   out          : [total_q, num_heads, head_size] in dtype, contiguous.
 *   lse          : float32 [num_heads, total_q] natural-log log-sum-exp of the
 *                  scaled logits each row saw, or NULL. A row that sees no key
 *                  gets out = 0 and lse = -inf.
 *   workspace    : >= pa_varlen_fwd_workspace_size(...) bytes, 256-byte aligned;
 *                  its contents need no initialisation and are scratch after the
 *                  call. One workspace must not be used by two calls in flight.
 */
pa_status pa_varlen_fwd(const void* q, int64_t q_token_stride, const void* key_cache,
                        const void* value_cache, int64_t cache_block_stride,
                        const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                        const int32_t* block_table, int bt_stride, int num_seqs, int total_q,
                        int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                        int head_size, int block_size, int num_blocks, float softmax_scale,
                        int causal, void* out, float* lse, void* workspace,
                        size_t workspace_bytes, int dtype, int32_t* dev_status, void* stream);

/*
 * pa_merge_attn_states -- LSE-weighted combine of two partial attention
 * results over disjoint key sets ([FA-vLLM] §6.3 step 3 and §8.2
 * merge_attn_states(prefix_out, suffix_out, prefix_lse, suffix_lse)).
 *
 *   prefix_out, suffix_out, out : [num_tokens, num_heads, head_size] in dtype, contiguous.
 *   prefix_lse, suffix_lse      : float32 [num_heads, num_tokens], natural log.
 *   out_lse                     : float32 [num_heads, num_tokens] or NULL.
 * With m = max(a, b), wa = e^(a-m), wb = e^(b-m):
 *   out = (wa*prefix_out + wb*suffix_out) / (wa + wb), out_lse = m + ln(wa + wb);
 * a row whose two LSEs are both -inf gets out = 0, out_lse = -inf.
 * out may alias prefix_out or suffix_out.
 */
pa_status pa_merge_attn_states(void* out, float* out_lse, const void* prefix_out,
                               const float* prefix_lse, const void* suffix_out,
                               const float* suffix_lse, int num_tokens, int num_heads,
                               int head_size, int dtype, void* stream);

/*
 * pa_merge_attn_states_n -- LSE-weighted combine of num_parts partial
 * attention results over disjoint key sets: the merge step of decode context
 * parallelism ([FA-vLLM] §9 and the DCP branch of §4: every rank attends over
 * its own KV shard, non-causal for decode, and the ranks' partial (out, lse)
 * are merged by LSE -- there by all-gather + reduce-scatter across GPUs; here
 * on one GPU, for ranks that are virtual), and the n-part form of
 * pa_merge_attn_states.
 *
 *   parts_out : dtype; part r is [num_tokens, num_heads, head_size] contiguous
 *               at parts_out + r * part_stride_out (elements, a multiple of 8,
 *               >= num_tokens * num_heads * head_size when num_parts > 1).
 *   parts_lse : float32; part r is [num_heads, num_tokens] at
 *               parts_lse + r * part_stride_lse (>= num_heads * num_tokens).
 *   out       : [num_tokens, num_heads, head_size] in dtype; may alias a part.
 *   out_lse   : float32 [num_heads, num_tokens] or NULL; must not overlap the
 *               parts' LSEs (PA_ERR_INVALID_ARG).
 * With m = max_r lse_r and w_r = e^(lse_r - m): out = sum_r w_r out_r /
 * sum_r w_r, out_lse = m + ln sum_r w_r (float32 throughout, out rounded to
 * dtype once). A row whose LSEs are all -inf gets out = 0, out_lse = -inf.
 * 1 <= num_parts <= PA_MERGE_N_MAX.
 *
 * A virtual-rank decode over R ranks is R pa_varlen_fwd calls (causal = 0),
 * one per rank with that rank's block table and key counts, writing into the
 * parts of one stacked buffer, followed by this merge.
 */
#define PA_MERGE_N_MAX 1024
pa_status pa_merge_attn_states_n(void* out, float* out_lse, const void* parts_out,
                                 int64_t part_stride_out, const float* parts_lse,
                                 int64_t part_stride_lse, int num_parts, int num_tokens,
                                 int num_heads, int head_size, int dtype, void* stream);

/* Workspace bytes pa_cascade_fwd needs (same arguments as the varlen query). */
size_t pa_cascade_fwd_workspace_size(int num_seqs, int total_q, int max_seqlen_q,
                                     int max_seqlen_k, int num_heads, int num_kv_heads,
                                     int head_size, int block_size, int sm_count);

/*
 * pa_cascade_fwd -- shared-prefix (cascade) attention ([FA-vLLM] §6.3):
 *   1. prefix pass: all total_q query tokens, as one non-causal segment,
 *      against the first common_prefix_len keys of block_table row 0;
 *   2. suffix pass: each sequence, causal, against its own keys from position
 *      common_prefix_len on (block_table[s, common_prefix_len/block_size:]);
 *   3. the two states merged by LSE as in pa_merge_attn_states.
 * The result equals pa_varlen_fwd(causal = 1) over the whole KV. Arguments as
 * pa_varlen_fwd plus common_prefix_len. Preconditions: common_prefix_len is a
 * multiple of block_size (else PA_ERR_INVALID_ARG); every row's first
 * common_prefix_len / block_size block_table entries equal row 0's; and
 * seqused_k[s] - q_len(s) >= common_prefix_len for every sequence, so every
 * query lies in its private suffix. A sequence that breaks the last rule sets
 * PA_DEV_CASCADE; its rows still follow the three steps literally (every
 * prefix key, then the causal suffix), which then differs from flat attention.
 * The shared-entries rule is not checked (row 0's pages are used).
 */
pa_status pa_cascade_fwd(const void* q, int64_t q_token_stride, const void* key_cache,
                         const void* value_cache, int64_t cache_block_stride,
                         const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                         const int32_t* block_table, int bt_stride, int num_seqs, int total_q,
                         int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                         int head_size, int block_size, int num_blocks, float softmax_scale,
                         int common_prefix_len, void* out, float* lse, void* workspace,
                         size_t workspace_bytes, int dtype, int32_t* dev_status, void* stream);

/*
 * pa_use_cascade_attention -- should a batch run as cascade attention?
 * ([FA-vLLM] §6.2, use_cascade_attention: a shared prefix of at least 256
 * tokens, at least 8 requests, no ALiBi / sliding window / local attention
 * and no DCP -- none of which this library has -- then cascade outright if
 * split-KV decoding is off, else whichever of the two is estimated faster.)
 * The pages leave the estimate open; this one compares bytes: flat attention
 * reads the shared prefix once per sequence, cascade reads it once and pays
 * a fixed cost for its extra pass and merge, so cascade is chosen when
 *   (num_seqs - 1) * common_prefix_len * num_kv_heads * head_size * 4 bytes
 *     > PA_CASCADE_FIXED_US * 1e-6 * PA_CASCADE_HBM_GBS * 1e9,
 * i.e. when re-reading the prefix would cost more than the extra pass.
 *   split_kv : 1 if the flat path may split keys over CTAs (pa_varlen_fwd
 *              does), 0 if not.
 * Writes 1 (cascade) or 0 (flat) to *use_cascade. Host only, no CUDA call.
 * PA_ERR_INVALID_ARG for negative sizes or a NULL use_cascade.
 */
#define PA_CASCADE_FIXED_US 20.0
#define PA_CASCADE_HBM_GBS 6500.0
pa_status pa_use_cascade_attention(int common_prefix_len, int num_seqs, int num_kv_heads,
                                   int head_size, int split_kv, int* use_cascade);

/*
 * New tokens' K/V for the update-and-attend entry points below: the
 * arguments of pa_reshape_and_cache that are not already arguments of the
 * attention call. key / value: [num_tokens, num_kv_heads, head_size] in dtype,
 * token t at key + t*key_token_stride; slot_mapping: int64 [num_tokens]
 * (slot < 0 skips the token). All device pointers, owned by the caller.
 */
typedef struct pa_kv_update {
  const void* key;
  const void* value;
  int64_t key_token_stride;
  int64_t value_token_stride;
  const int64_t* slot_mapping;
  int num_tokens;
} pa_kv_update;

/*
 * pa_varlen_fwd_with_update / pa_cascade_fwd_with_update -- one serving step
 * ([FA-vLLM] §4.2: the forward pass first writes the step's new K/V into the
 * paged cache by slot_mapping, then attends): the same result as
 * pa_reshape_and_cache(update, key_cache, value_cache, ...) followed by
 * pa_varlen_fwd / pa_cascade_fwd with the remaining arguments, on the same
 * stream. In one call the planner and the scatter run concurrently (the
 * planner reads only the sequence metadata), and the attention kernels start
 * once both have finished. update may be NULL or have num_tokens = 0 (then
 * these equal pa_varlen_fwd / pa_cascade_fwd). The cache arguments
 * (cache_block_stride, num_kv_heads, head_size, block_size, num_blocks) and
 * dev_status serve both parts; the update's arguments are checked like
 * pa_reshape_and_cache's before anything is launched.
 */
pa_status pa_varlen_fwd_with_update(const pa_kv_update* update, const void* q,
                                    int64_t q_token_stride, void* key_cache, void* value_cache,
                                    int64_t cache_block_stride, const int32_t* cu_seqlens_q,
                                    const int32_t* seqused_k, const int32_t* block_table,
                                    int bt_stride, int num_seqs, int total_q, int max_seqlen_q,
                                    int max_seqlen_k, int num_heads, int num_kv_heads,
                                    int head_size, int block_size, int num_blocks,
                                    float softmax_scale, int causal, void* out, float* lse,
                                    void* workspace, size_t workspace_bytes, int dtype,
                                    int32_t* dev_status, void* stream);
pa_status pa_cascade_fwd_with_update(const pa_kv_update* update, const void* q,
                                     int64_t q_token_stride, void* key_cache, void* value_cache,
                                     int64_t cache_block_stride, const int32_t* cu_seqlens_q,
                                     const int32_t* seqused_k, const int32_t* block_table,
                                     int bt_stride, int num_seqs, int total_q, int max_seqlen_q,
                                     int max_seqlen_k, int num_heads, int num_kv_heads,
                                     int head_size, int block_size, int num_blocks,
                                     float softmax_scale, int common_prefix_len, void* out,
                                     float* lse, void* workspace, size_t workspace_bytes,
                                     int dtype, int32_t* dev_status, void* stream);

/*
 * pa_varlen_fwd_noalloc -- pa_varlen_fwd for callers that cannot allocate
 * device memory, so cannot provide a workspace: for example a serving engine
 * whose allocator reserved all device memory for its page pool at start-up,
 * or a latency-critical path where cudaMalloc's implicit device
 * synchronisation is not acceptable. The web pages have no counterpart to
 * this entry point; it only changes where the scratch lives.
 *
 * Arguments, layouts and results are those of pa_varlen_fwd without
 * workspace / workspace_bytes. The scratch is a fixed, library-owned
 * PA_NOALLOC_SCRATCH_BYTES (32 MiB) device buffer: every GPU that loads
 * libpa.so holds it until the process exits. A problem whose
 * pa_varlen_fwd_workspace_size exceeds it is rejected with
 * PA_ERR_NOALLOC_LIMIT before anything is launched. The function never calls
 * cudaMalloc, cudaFree or any allocating routine.
 *  - The first call on a device looks up that buffer's device address (with
 *    the device current) and caches it with the device's current context;
 *    make that first call before any stream capture on the device. After
 *    cudaDeviceReset (a new context) the next call looks it up again, so
 *    make that call before any capture too. A failed lookup returns
 *    PA_ERR_CUDA and leaves no CUDA error pending.
 *  - Every call uses the same buffer, which keeps the previous call's
 *    contents; the kernels rewrite everything they read before reading it, so
 *    nothing needs clearing. Calls that overlap on the GPU (two streams, or
 *    two host threads without ordering) race on the buffer: serialise them.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)

pa_status pa_varlen_fwd_noalloc(const void* q, int64_t q_token_stride, const void* key_cache,
                                const void* value_cache, int64_t cache_block_stride,
                                const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                                const int32_t* block_table, int bt_stride, int num_seqs,
                                int total_q, int max_seqlen_q, int max_seqlen_k, int num_heads,
                                int num_kv_heads, int head_size, int block_size, int num_blocks,
                                float softmax_scale, int causal, void* out, float* lse, int dtype,
                                int32_t* dev_status, void* stream);

/*
 * FP8 (e4m3) KV cache ([FA/FI] 役割 and 境界と失敗: FlashInfer and FA3 accept
 * an fp8 / fp8_e4m3 KV cache with per-head quant scales; [FA-vLLM] §10 lists an
 * FP8 KV cache among the backends' features).
 *
 * The pools hold one byte per element: the OCP 8-bit floating point "E4M3"
 * format (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest
 * finite value 448, no infinities, S.1111.111 is NaN). A stored byte c of KV
 * head h means the value e4m3(c) * scale[h]. Writes store
 * e4m3(x / scale[h]): x is the bf16 or f16 input widened to float32, the division
 * is IEEE float32 (correctly rounded), the result is rounded to the nearest
 * e4m3 value (ties to even) and saturates at +-448 (a NaN stays NaN).
 * Attention computes exactly the 2-byte pools' definition on the dequantized
 * keys and values e4m3(c) * scale[h], with float32 accumulation. Segments
 * of more than 32 packed query rows (prefill) run on the tensor-core kernel:
 * q.k on the e4m3 tensor MMA straight from the stored key bytes, p.v on the
 * f16 MMA with each e4m3 V tile widened to f16 in shared memory (exact).
 * Shorter segments run on the split-KV kernel: items of at most 8 packed
 * rows (decode with GQA <= 8) take q.k on the e4m3 MMA too, wider ones form
 * q.k from f16 q (there |q| must stay below 65504). Wherever q.k is on the
 * e4m3 MMA, q is taken as two e4m3 terms after a power-of-two row scale
 * (exact for every element of at least 2^-9 of its row's largest).
 * Layout: the NHD pools of pa_reshape_and_cache with 1-byte elements;
 * cache_block_stride is in elements (= bytes) and a multiple of 16.
 * head_size must be 128 (PA_ERR_UNSUPPORTED otherwise).
 */
typedef struct pa_kv_fp8 {
  const float* k_scale; /* device float32 [num_kv_heads], finite and > 0 (not checked) */
  const float* v_scale; /* device float32 [num_kv_heads], finite and > 0 (not checked) */
} pa_kv_fp8;

/*
 * pa_reshape_and_cache_fp8 -- pa_reshape_and_cache into e4m3 pools: key /
 * value are bf16 or f16 rows as there (dtype); each element is quantized
 * with its KV head's scale as described above. scales must be non-NULL with
 * both pointers 4-byte aligned (PA_ERR_INVALID_ARG).
 */
pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, int64_t key_token_stride,
                                   int64_t value_token_stride, void* key_cache, void* value_cache,
                                   int64_t cache_block_stride, const int64_t* slot_mapping,
                                   int num_tokens, int num_kv_heads, int head_size,
                                   int block_size, int num_blocks, const pa_kv_fp8* scales,
                                   int dtype, int32_t* dev_status, void* stream);

/* Workspace bytes of pa_varlen_fwd_fp8kv / pa_cascade_fwd_fp8kv (0 if invalid). */
size_t pa_varlen_fwd_fp8kv_workspace_size(int num_seqs, int total_q, int max_seqlen_q,
                                          int max_seqlen_k, int num_heads, int num_kv_heads,
                                          int head_size, int block_size, int sm_count);
size_t pa_cascade_fwd_fp8kv_workspace_size(int num_seqs, int total_q, int max_seqlen_q,
                                           int max_seqlen_k, int num_heads, int num_kv_heads,
                                           int head_size, int block_size, int sm_count);

/*
 * pa_varlen_fwd_fp8kv / pa_cascade_fwd_fp8kv -- pa_varlen_fwd_with_update /
 * pa_cascade_fwd_with_update over e4m3 pools: the optional update (NULL or
 * num_tokens = 0 for none) is quantized into the pools as by
 * pa_reshape_and_cache_fp8, then the attention reads the dequantized cache.
 * q, out and lse are as in the other entry points (dtype PA_BF16 or PA_F16).
 */
pa_status pa_varlen_fwd_fp8kv(const pa_kv_update* update, const void* q, int64_t q_token_stride,
                              void* key_cache, void* value_cache, int64_t cache_block_stride,
                              const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                              const int32_t* block_table, int bt_stride, int num_seqs,
                              int total_q, int max_seqlen_q, int max_seqlen_k, int num_heads,
                              int num_kv_heads, int head_size, int block_size, int num_blocks,
                              float softmax_scale, int causal, const pa_kv_fp8* scales, void* out,
                              float* lse, void* workspace, size_t workspace_bytes, int dtype,
                              int32_t* dev_status, void* stream);
pa_status pa_cascade_fwd_fp8kv(const pa_kv_update* update, const void* q,
                               int64_t q_token_stride, void* key_cache, void* value_cache,
                               int64_t cache_block_stride, const int32_t* cu_seqlens_q,
                               const int32_t* seqused_k, const int32_t* block_table,
                               int bt_stride, int num_seqs, int total_q, int max_seqlen_q,
                               int max_seqlen_k, int num_heads, int num_kv_heads, int head_size,
                               int block_size, int num_blocks, float softmax_scale,
                               int common_prefix_len, const pa_kv_fp8* scales, void* out,
                               float* lse, void* workspace, size_t workspace_bytes, int dtype,
                               int32_t* dev_status, void* stream);

/*
 * Options of the pa_*_fwd_ex entry points (NULL, or a NULL field, means the
 * default).
 *   sinks : attention sinks ([FA-vLLM] §1.2 and §1.3: the s_aux learnable sink
 *           token of FA3/FA4) -- device float32 [num_heads], one logit per
 *           query head in the units of softmax_scale * q.k, 4-byte aligned.
 *           Each acts as one more key of that logit and value zero: with
 *           s_j = softmax_scale * q.k_j over the visible keys,
 *           out = sum_j e^(s_j) v_j / (sum_j e^(s_j) + e^(sink)) and
 *           lse = ln(sum_j e^(s_j) + e^(sink)); a row with no visible key gets
 *           out = 0 and lse = sink.
 *   fp8   : NULL for 2-byte pools (dtype), else the pools hold e4m3 bytes with these
 *           scales (as in pa_varlen_fwd_fp8kv; workspace then per
 *           pa_*_fwd_fp8kv_workspace_size).
 */
typedef struct pa_attn_opts {
  const float* sinks;
  const pa_kv_fp8* fp8;
} pa_attn_opts;

/*
 * pa_varlen_fwd_ex / pa_cascade_fwd_ex -- pa_varlen_fwd_with_update /
 * pa_cascade_fwd_with_update with options (opts may be NULL: then they are
 * those entry points exactly).
 */
pa_status pa_varlen_fwd_ex(const pa_kv_update* update, const void* q, int64_t q_token_stride,
                           void* key_cache, void* value_cache, int64_t cache_block_stride,
                           const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                           const int32_t* block_table, int bt_stride, int num_seqs, int total_q,
                           int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                           int head_size, int block_size, int num_blocks, float softmax_scale,
                           int causal, const pa_attn_opts* opts, void* out, float* lse,
                           void* workspace, size_t workspace_bytes, int dtype,
                           int32_t* dev_status, void* stream);
pa_status pa_cascade_fwd_ex(const pa_kv_update* update, const void* q, int64_t q_token_stride,
                            void* key_cache, void* value_cache, int64_t cache_block_stride,
                            const int32_t* cu_seqlens_q, const int32_t* seqused_k,
                            const int32_t* block_table, int bt_stride, int num_seqs,
                            int total_q, int max_seqlen_q, int max_seqlen_k, int num_heads,
                            int num_kv_heads, int head_size, int block_size, int num_blocks,
                            float softmax_scale, int common_prefix_len, const pa_attn_opts* opts,
                            void* out, float* lse, void* workspace, size_t workspace_bytes,
                            int dtype, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
