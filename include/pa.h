/*
 * pa.h -- C ABI of the GB300 (sm_103a) paged-KV attention library (libpa.so).
 *
 * The operations are those of vLLM-style paged attention as the source pages
 * define them:
 *   - the K/V pool: per layer one K and one V tensor of shape
 *     [num_blocks, block_size, num_kv_heads, head_dim], row-major
 *     ("分页 KV Cache", §实现 and the PagedKVCache class of its paged.py);
 *   - a token at position p of a request lives in logical block
 *     p / block_size at offset p % block_size; the request's block table maps
 *     the logical block to a physical one, and the token's slot is
 *     physical_block * block_size + offset ("分页 KV Cache", §块表与 slot
 *     mapping; "PagedAttention：分页内存管理", §block_table translation);
 *   - attention reads each request's K/V through its block table, with the
 *     new tokens at the end of the context and a causal mask ("分页 KV
 *     Cache", §分页注意力 and paged_attention; "aiqz.cc PagedAttention",
 *     §工程实现要点: per-block partial softmax merged online);
 *   - copy-on-write copies a shared block into a fresh one before a write
 *     ("分页 KV Cache", exercise 2; "KV cache：容量推导、分页与回收",
 *     §共享前缀后为什么需要引用计数).
 *
 * Conventions for every entry point:
 *   - Pointers named as device pointers are device memory owned by the
 *     caller, contiguous, row-major, 16-byte aligned where noted.  The
 *     library allocates nothing and keeps no pointer after the call returns.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream) on the current device.
 *   - Argument errors are returned synchronously, before anything is
 *     enqueued: PA_ERR_INVALID_ARG (bad size, null pointer, misalignment),
 *     PA_ERR_UNSUPPORTED (a valid but unsupported shape or dtype),
 *     PA_ERR_WORKSPACE (workspace too small).  PA_ERR_CUDA reports a
 *     launch failure.  PA_ERR_INDEX is returned only in check mode
 *     (pa_set_check_mode), which copies the index arrays to the host and
 *     validates them before launching; without check mode an out-of-range
 *     block id, slot or length is undefined behaviour, as with tensor
 *     indexing in the pages' reference code.  pa_last_error() gives a
 *     human-readable reason for the last non-OK status of the calling thread.
 *   - Block-table rows are padded to max_blocks; entries at or past
 *     ceil(len / block_size) are never read.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,
    PA_ERR_UNSUPPORTED = 2,
    PA_ERR_INDEX = 3,
    PA_ERR_WORKSPACE = 4,
    PA_ERR_CUDA = 5,
    PA_ERR_TIMEOUT = 6
} pa_status;

/* PA_FP8_E4M3: a quantized cache of 1-byte E4M3 codes (the OCP 8-bit
 * floating-point format: 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, largest finite value 448, S.1111.111 = NaN).  Accepted as the pool
 * type of pa_copy_blocks and pa_swap_blocks (which move bytes); the FP8
 * entry points below take it implicitly. */
typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_F16 = 2, PA_FP8_E4M3 = 3 } pa_dtype;

/* Library options (pa_set_option).  Global to the process, not thread-safe
 * against concurrent calls. */
typedef enum {
    /* 1: validate index arrays on the host before each launch (synchronises
     * the stream).  0 (default): no validation. */
    PA_OPT_CHECK_MODE = 0,
    /* Decode kernel: 0 automatic (default), 1 the CUDA-core kernel, 2 the
     * tensor-core kernel (PA_ERR_UNSUPPORTED where it does not apply). */
    PA_OPT_DECODE_KERNEL = 1,
    /* Number of CTAs of the tensor-core decode kernel's balanced split;
     * 0 (default) picks one per resident slot of the device. */
    PA_OPT_DECODE_CTAS = 2,
    /* Varlen kernel: 0 automatic (default: the tcgen05 kernel where it
     * applies, else the CUDA-core kernel), 1 the CUDA-core kernel, 2 the
     * tcgen05 (tensor-memory) kernel (PA_ERR_UNSUPPORTED where it does not
     * apply). */
    PA_OPT_VARLEN_KERNEL = 3,
    /* Code-cache decode, head_dim 128: work the two tiles of a pipeline stage
     * that belong to one (sequence, KV head) as one 32-token step (one
     * softmax reduction, two independent score chains).  0 automatic
     * (default: when max_context > 2048, where sequences are long enough
     * that most stages hold two tiles of one unit), 1 never, 2 always.
     * Results agree within the tolerance either way. */
    PA_OPT_FP8_PAIR_STEP = 4
} pa_option;

PA_API const char* pa_status_string(int status);
/* Reason for the last non-OK status returned on the calling thread. */
PA_API const char* pa_last_error(void);
PA_API pa_status pa_set_option(int option, int64_t value);
PA_API int64_t pa_get_option(int option);
/* Shorthand for pa_set_option(PA_OPT_CHECK_MODE, on). */
PA_API pa_status pa_set_check_mode(int on);

/* Device-side status word: kernels that wait on a barrier give up after a
 * bounded number of polls, set a bit here and return (PA_ERR_TIMEOUT).
 * Reads (and with clear != 0 resets) it for the current device; synchronises
 * the device. */
PA_API pa_status pa_device_status(int clear);

/* Exercises that failure path without a fault (library self-test; the pages
 * have no counterpart): one CTA waits on a shared-memory barrier that nothing
 * completes, with the same bounded wait the decode kernel uses, gives up
 * after `polls` polls (1 .. 2^20), sets the timeout bit and returns; a
 * following pa_device_status reports PA_ERR_TIMEOUT (and clears it on
 * request).  Nothing else is touched and the context stays usable. */
PA_API pa_status pa_selftest_wait_timeout(int32_t polls, void* stream);

/*
 * pa_slot_mapping -- slot of each new token.
 *   slot_out[i] = block_tables[seq_idx[i] * max_blocks + positions[i] / block_size]
 *                 * block_size + positions[i] % block_size
 * ("分页 KV Cache", slot_mapping_for; "PagedAttention：分页内存管理",
 * translate_slot).  positions[i] < 0 marks a padding token: slot_out[i] = -1.
 *   block_tables: device int32 [num_seqs, max_blocks]
 *   seq_idx:      device int32 [n], 0 <= seq_idx[i] < num_seqs
 *   positions:    device int64 [n]
 *   slot_out:     device int64 [n] (written)
 */
PA_API pa_status pa_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks,
                          const int32_t* seq_idx, const int64_t* positions, int64_t n,
                          int32_t block_size, int64_t* slot_out, void* stream);

/*
 * pa_write_kv -- scatter new tokens' K and V rows into the pool.
 * The cache viewed as [num_blocks * block_size, num_kv_heads * head_dim]
 * rows; row slot_mapping[i] of k_cache receives k[i], of v_cache v[i]
 * ("分页 KV Cache", PagedKVCache.write).  A negative slot skips token i
 * (padding).  Slots must be distinct (check mode rejects duplicates).
 *   k, v:          device [n, num_kv_heads, head_dim] of dtype, 16-byte aligned
 *   slot_mapping:  device int64 [n]
 *   k_cache, v_cache: device [num_blocks, block_size, num_kv_heads, head_dim]
 * Requires num_kv_heads * head_dim * sizeof(dtype) to be a multiple of 16.
 * Bit-exact: bytes are moved, never converted.
 */
PA_API pa_status pa_write_kv(const void* k, const void* v, const int64_t* slot_mapping, int64_t n,
                      void* k_cache, void* v_cache, int32_t num_blocks, int32_t block_size,
                      int32_t num_kv_heads, int32_t head_dim, int dtype, void* stream);

/*
 * pa_write_kv_fp8 -- the quantizing form of pa_write_kv, for a quantized
 * cache.  The pages name a quantized cache (量化缓存) as one that changes the
 * per-token KV size ("KV cache：容量推导、分页与回收", §输入放得下，输出还要留空间) and give
 * no method; the reading implemented here: each (token, KV head) row x of
 * k[i] (and of v[i]) is stored as E4M3 codes with one fp32 scale,
 *   scale = max|x| / 448   (1 for an all-zero row),
 *   code  = E4M3(x / scale), nearest with ties to even, held at +-448,
 * the maximum and the division taken in fp32 (IEEE).  Codes go to row
 * slot_mapping[i] of the code pools exactly where pa_write_kv puts a row; the
 * scale of KV head h goes to
 *   scales[(slot / block_size) * num_kv_heads + h) * block_size + slot % block_size],
 * i.e. scales are laid out [num_blocks, num_kv_heads, block_size] so the 16
 * scales a decode tile needs are contiguous.  A negative slot skips token i;
 * slots must be distinct (check mode rejects duplicates and out-of-pool
 * slots).  Bit-exact against that definition.
 *   k, v:              device [n, num_kv_heads, head_dim] of dtype (PA_F32/BF16/F16), 16-byte aligned
 *   slot_mapping:      device int64 [n]
 *   k_codes, v_codes:  device uint8 [num_blocks, block_size, num_kv_heads, head_dim], 16-byte aligned
 *   k_scales, v_scales: device fp32 [num_blocks, num_kv_heads, block_size]
 * head_dim <= 256.
 */
PA_API pa_status pa_write_kv_fp8(const void* k, const void* v, const int64_t* slot_mapping, int64_t n,
                                 void* k_codes, void* v_codes, float* k_scales, float* v_scales, int32_t num_blocks,
                                 int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int dtype,
                                 void* stream);

/*
 * pa_copy_blocks -- copy-on-write block copies.
 * For each layer l and pair p: block block_pairs[2p+1] of k_caches[l] and of
 * v_caches[l] receives a copy of block block_pairs[2p] (all block_size
 * slots).  k_caches / v_caches are HOST arrays of num_layers device
 * pointers (1 <= num_layers <= PA_MAX_LAYERS).  A destination must not be
 * the source or destination of another pair of the same call (check mode
 * rejects that); otherwise the pairs run in any order.
 *   block_pairs: device int64 [num_pairs, 2] (src, dst)
 * dtype may be PA_FP8_E4M3 (a quantized cache's code pools); its scale
 * pools [num_blocks, num_kv_heads, block_size] are copied by a second call
 * with dtype PA_F32 and head_dim 1.
 */
#define PA_MAX_LAYERS 128
PA_API pa_status pa_copy_blocks(void* const* k_caches, void* const* v_caches, int32_t num_layers,
                         const int64_t* block_pairs, int32_t num_pairs, int32_t num_blocks,
                         int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int dtype,
                         void* stream);

/*
 * pa_swap_blocks -- move whole blocks between two pools, e.g. the device
 * pool and a host pool when sequences are preempted and resumed (the xxqk.cn
 * PagedAttention article, §显存不够时的调度: evicted blocks go to CPU memory
 * and come back; small blocks make this many small transfers).  For each
 * layer l and pair p: block block_pairs[2p+1] of dst_k[l] / dst_v[l]
 * receives block block_pairs[2p] of src_k[l] / src_v[l] (all block_size
 * slots).  src_* and dst_* are HOST arrays of num_layers pointers; each
 * pointer is device memory or pinned/registered host memory (the GPU reads
 * or writes host pools directly, over NVLink-C2C on GB300); block_pairs is
 * device or pinned host memory, int64 [num_pairs, 2] (src, dst).  Any other
 * memory is PA_ERR_INVALID_ARG.  Destinations must be distinct and the two
 * pools distinct (or the pairs' source and destination sets disjoint);
 * check mode rejects out-of-range ids and repeated destinations.  Enqueued
 * on `stream`; host pools must stay allocated until it completes.
 * Bit-exact.
 */
PA_API pa_status pa_swap_blocks(void* const* src_k, void* const* src_v, void* const* dst_k,
                                void* const* dst_v, int32_t num_layers, const int64_t* block_pairs,
                                int32_t num_pairs, int32_t src_num_blocks, int32_t dst_num_blocks,
                                int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int dtype,
                                void* stream);

/*
 * pa_decode -- one query per sequence over its paged context.
 * For sequence s and query head h (KV head kv = h / (num_heads / num_kv_heads),
 * the repeat_interleave grouping of the handbook's paged_attention):
 *   out[s, h] = softmax(scale * q[s, h] . K_s[0:L]^T) . V_s[0:L],  L = context_lens[s]
 * where K_s / V_s are read through block_tables[s].  This is the num_new = 1
 * case of pa_varlen (the query is the last position, so it sees all L keys).
 * The context is split across CTAs by a length-balanced partition and the
 * partial softmax states are merged by their log-sum-exp; the partition
 * depends only on the lengths, so relabelling physical blocks gives
 * bit-identical output.  context_lens[s] == 0 gives a zero row.
 *   out, q:       device [num_seqs, num_heads, head_dim] of dtype (16-byte aligned)
 *   k_cache, v_cache: device [num_blocks, block_size, num_kv_heads, head_dim]
 *   block_tables: device int32 [num_seqs, max_blocks]
 *   context_lens: device int32 [num_seqs], each <= max_context
 *   workspace:    device scratch of at least pa_decode_workspace_size(...) bytes
 *                 (may be NULL when that size is 0), 16-byte aligned; its
 *                 content on entry does not matter.
 * Accumulation is fp32 for every dtype.  bf16/f16 with head_dim 64/128/256
 * and at most 16 query heads per KV head run on the tensor cores at any
 * block size (TMA boxes for 8 and multiples of 16 up to 256, a row-by-row
 * gather otherwise); the rest on the CUDA-core kernel, which reads each K/V
 * row once for up to 8 query heads of a KV head.
 */
PA_API size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, int32_t max_context, int dtype);
PA_API pa_status pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                    int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t num_blocks, int32_t block_size, int32_t max_context, float scale,
                    int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_fp8 -- pa_decode over a quantized cache (see pa_write_kv_fp8):
 * a key or value element is its code's value times its (token, KV head)
 * row's scale, and out is the decode attention of pa_decode over those
 * values.  The cache moves half the bytes of a 16-bit cache.  On the
 * tensor-core path (bf16/f16 q, head_dim 128 or 256, block_size 8 or a
 * multiple of 16 up to 256, at most 16 query heads per KV head) codes are
 * converted exactly to f16, q enters the mma as f16(q * scale * log2 e) and
 * each softmax weight times its value scale as f16; other shapes and fp32 q
 * run on the CUDA-core kernel in fp32.  Requires |q * scale| < 45000 on the
 * tensor-core path (the f16 range).
 *   out, q:            device [num_seqs, num_heads, head_dim] of dtype (PA_F32/BF16/F16)
 *   k_codes, v_codes:  device uint8 [num_blocks, block_size, num_kv_heads, head_dim]
 *   k_scales, v_scales: device fp32 [num_blocks, num_kv_heads, block_size], 16-byte aligned
 *   workspace:         pa_decode_fp8_workspace_size(...) bytes
 * The other arguments, the error behaviour and the split are pa_decode's.
 */
PA_API size_t pa_decode_fp8_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t block_size, int32_t max_context, int dtype);
PA_API pa_status pa_decode_fp8(void* out, const void* q, const void* k_codes, const void* v_codes,
                               const float* k_scales, const float* v_scales, const int32_t* block_tables,
                               int32_t max_blocks, const int32_t* context_lens, int32_t num_seqs, int32_t num_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                               int32_t max_context, float scale, int dtype, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * pa_decode_append -- one generation step of a decode batch in one call:
 * for each sequence s with L = context_lens[s] >= 1 (L counts the new
 * token), the new token's rows k_new[s], v_new[s] are written to the slot of
 * position L-1, block_tables[s][(L-1) / block_size] * block_size +
 * (L-1) % block_size ("分页 KV Cache", §块表与 slot mapping and
 * PagedKVCache.write), and out[s] is the decode attention over positions
 * 0..L-1 exactly as pa_decode computes it after that write ("分页 KV Cache",
 * §分页注意力: the step writes the new K/V, then attends).  Equivalent to
 * pa_slot_mapping + pa_write_kv + pa_decode; on the tensor-core path it is
 * one kernel launch.  Sequences with L = 0 get a zero row and no write.
 *   k_new, v_new: device [num_seqs, num_kv_heads, head_dim] of dtype, 16-byte aligned
 *   k_cache, v_cache: written at one slot per sequence (the other arguments
 *   as for pa_decode, same workspace size).
 */
PA_API pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                                  void* k_cache, void* v_cache, const int32_t* block_tables,
                                  int32_t max_blocks, const int32_t* context_lens, int32_t num_seqs,
                                  int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t num_blocks, int32_t block_size, int32_t max_context, float scale,
                                  int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_append_fp8 -- pa_decode_append over a quantized cache: each
 * sequence's new rows k_new[s], v_new[s] (of dtype, the query type) are
 * quantized as pa_write_kv_fp8 does it into the slot of position L-1 (codes
 * and scales), and out[s] is pa_decode_fp8 over positions 0..L-1 after that
 * write ("分页 KV Cache", §分页注意力: the step writes the new K/V, then
 * attends).  One kernel launch on the tensor-core path with head_dim 128;
 * otherwise a quantizing write kernel, then the decode.  Sequences with
 * L = 0 get a zero row and no write.  Same workspace as pa_decode_fp8.
 */
PA_API pa_status pa_decode_append_fp8(void* out, const void* q, const void* k_new, const void* v_new,
                                      void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                                      const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                                      int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t num_blocks, int32_t block_size, int32_t max_context, float scale,
                                      int dtype, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_varlen -- the handbook's paged_attention: a batch of requests, each
 * with seq_lens[i] tokens of context after this step of which the last
 * n_i = cu_seqlens_q[i+1] - cu_seqlens_q[i] are new; request i's queries
 * are rows cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1 of q.  New token j of
 * request i is at position seq_lens[i] - n_i + j and, with causal != 0,
 * attends to positions 0..that position; with causal == 0 to all
 * seq_lens[i] positions.  Decode rows (n_i = 1) and prefill chunks mix
 * freely in one call.  bf16/f16 with head_dim 64, 128 or 256, at most 128
 * query heads per KV head and block_size 8 or a multiple of 16 up to 256
 * (head_dim 256: a multiple of 16) run on the tcgen05 (tensor-memory)
 * kernel; the rest on the CUDA-core kernel.
 *   out, q:       device [total_q, num_heads, head_dim] of dtype (16-byte aligned)
 *   cu_seqlens_q: device int32 [num_seqs + 1], cu_seqlens_q[0] = 0,
 *                 non-decreasing, cu_seqlens_q[num_seqs] = total_q
 *   seq_lens:     device int32 [num_seqs], n_i <= seq_lens[i] <= max_context
 *   max_q:        upper bound of n_i over the batch
 *   workspace:    optional device scratch of pa_varlen_workspace_size(...)
 *                 bytes (16-byte aligned; caller-owned, contents need no
 *                 initialisation).  Given, the tensor-core kernel first lists
 *                 its work longest first (a one-CTA plan kernel) and runs it
 *                 in that order; NULL (or 0 bytes) runs it in request order.
 *                 The outputs are the same either way.  A non-NULL workspace
 *                 smaller than the size returns PA_ERR_WORKSPACE.  The size
 *                 is 0 where the CUDA-core kernel runs (fp32, other head
 *                 dims, PA_OPT_VARLEN_KERNEL = 1).
 */
PA_API size_t pa_varlen_workspace_size(int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_heads,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                int32_t max_context, int dtype);
PA_API pa_status pa_varlen(void* out, const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                    const int32_t* cu_seqlens_q, int32_t num_seqs, int32_t total_q, int32_t max_q,
                    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                    int32_t block_size, int32_t max_context, float scale, int causal, int dtype,
                    void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_varlen_fp8 -- pa_varlen over a quantized cache (see pa_write_kv_fp8):
 * the handbook's paged_attention ("分页 KV Cache", §分页注意力) with each key
 * and value element its code's value times its (token, KV head) row's scale
 * (the quantized cache of "KV cache：容量推导、分页与回收", §输入放得下，输出
 * 还要留空间).  Prefill chunks and decode rows mix as in pa_varlen; causal
 * as there.  bf16/f16 queries with head_dim 128 and block_size 8 or a
 * multiple of 16 up to 256 run on the tcgen05 kernel: code tiles are turned
 * into f16 code x scale in shared memory and the MMAs run in f16 (q, and
 * the keys and values, must lie inside the f16 range); the rest runs on the
 * CUDA-core kernel (fp32 arithmetic, any head_dim up to 256 and any block
 * size).
 *   out, q:             device [total_q, num_heads, head_dim] of dtype (PA_F32/BF16/F16)
 *   k_codes, v_codes:   device uint8 [num_blocks, block_size, num_kv_heads, head_dim]
 *   k_scales, v_scales: device fp32 [num_blocks, num_kv_heads, block_size], 16-byte aligned
 *   workspace:          optional, pa_varlen_fp8_workspace_size(...) bytes: as
 *                       for pa_varlen, the tcgen05 kernel then runs its work
 *                       longest first
 * The other arguments and the error behaviour are pa_varlen's.
 */
PA_API size_t pa_varlen_fp8_workspace_size(int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_heads,
                                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                           int32_t max_context, int dtype);
PA_API pa_status pa_varlen_fp8(void* out, const void* q, const void* k_codes, const void* v_codes,
                               const float* k_scales, const float* v_scales, const int32_t* block_tables,
                               int32_t max_blocks, const int32_t* seq_lens, const int32_t* cu_seqlens_q,
                               int32_t num_seqs, int32_t total_q, int32_t max_q, int32_t num_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks, int32_t block_size,
                               int32_t max_context, float scale, int causal, int dtype, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device
 * memory when they run it: a runtime or plugin host that hands out all
 * device memory from its own pool and forbids cudaMalloc in its callbacks, a
 * latency-critical loop that cannot afford an allocation's possible device
 * synchronisation, or code with no allocator at hand.  The pages have no
 * counterpart; it exists for those callers only.
 * Same arguments and result as pa_decode (tensor-core cases: bf16/f16,
 * head_dim 64/128/256, any block_size, at most 16 query heads per KV head;
 * others return PA_ERR_UNSUPPORTED), but no
 * workspace: the split-KV scratch
 * is one library-owned device array of 8 MiB per device, held from load
 * until process exit.  A problem whose scratch (pa_decode_workspace_size
 * with default options) exceeds 8 MiB returns PA_ERR_WORKSPACE before
 * anything is enqueued.  The call allocates nothing.  The first call with a
 * device current looks up that device's array address (again after the
 * device's context was replaced, e.g. by cudaDeviceReset); make it before
 * any stream capture.  All calls on a device share the array: calls whose
 * kernels overlap on the GPU race and must be ordered by the caller.
 * Check mode (PA_OPT_CHECK_MODE) applies as for pa_decode: lengths and
 * tables are copied to the host and validated (PA_ERR_INDEX) before launch.
 * The array need not start at zero, and no call reads what an earlier one
 * left in it (each launch writes every split record its merge reads, and
 * the merge finds them from the lengths alone), so it never needs clearing -- not even after a bounded wait
 * ran out (PA_ERR_TIMEOUT).
 */
PA_API pa_status pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks,
                                   const int32_t* context_lens, int32_t num_seqs, int32_t num_heads,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                                   int32_t block_size, int32_t max_context, float scale, int dtype,
                                   void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
