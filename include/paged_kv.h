/*
 * paged_kv.h -- C ABI of the GB300 paged KV cache library (libpaged_kv.so).
 *
 * The problem these calls solve is the one stated by the pages:
 *   - the physical KV cache is laid out [num_blocks, block_size, H_kv, d]
 *     ("KVCache 优化技能" skill note, 模式二 and §3.1);
 *   - new K/V rows are written through slot_mapping, one slot per new token,
 *     slot = block_table[b, pos / block_size] * block_size + pos % block_size
 *     (same note §3.1 / §3.3; "KV Cache 管理设计文档" §4.2.2 prepare_slot_mapping);
 *   - attention reads each sequence's keys through block_table with per-sequence
 *     lengths (actual_seq_lengths_kv), for GQA, sliding windows whose expired
 *     table entries hold a null block, causal prefill, and the absorbed MLA form.
 *
 * Conventions shared by every call:
 *   - Return value: PKV_OK (0) or a negative PKV_ERR_* code. On error nothing was
 *     launched and pkv_last_error() (thread-local) holds a one-line reason.
 *   - Device calls take device pointers owned by the caller and run
 *     asynchronously on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     The library never allocates, frees or synchronises device memory; scratch
 *     space is a caller-provided `workspace` of at least the size the matching
 *     *_workspace_size() call returns, 256-byte aligned.
 *   - Element types: q, caches and new rows are bf16 (raw 16-bit storage);
 *     block tables, slot mappings and lengths are int32. `out_dtype` selects a
 *     bf16 (PKV_BF16, round-to-nearest-even) or fp32 (PKV_F32) output.
 *   - `scale` has no default: callers pass it (the pages warn that a softmax
 *     scale silently falling back to 1.0 ruins accuracy, standalone guide FA
 *     v1/v2 parameter table).
 *   - `dev_status` (nullable) is a device int the kernels set to a nonzero
 *     PKV_DEV_* bit mask when they meet a bad table entry, slot or length; the
 *     offending access is skipped (never performed). The caller zeroes it.
 *   - Tensor-memory-accelerator (TMA) reads need 16-byte aligned base pointers
 *     and row strides; every pointer below must be 16-byte aligned.
 */
#ifndef PAGED_KV_H
#define PAGED_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG (-1)   /* null pointer, bad size, misaligned pointer   */
#define PKV_ERR_UNSUPPORTED (-2)   /* a shape this build does not implement        */
#define PKV_ERR_WORKSPACE (-3)     /* workspace missing or too small               */
#define PKV_ERR_LAUNCH (-4)        /* CUDA launch or driver call failed             */
#define PKV_ERR_OUT_OF_BLOCKS (-5) /* pool cannot satisfy an all-or-nothing request */
#define PKV_ERR_DOUBLE_FREE (-6)   /* freeing a free block or the null block        */

/* bits of *dev_status */
#define PKV_DEV_BAD_SLOT 1         /* slot_mapping entry >= num_blocks * block_size  */
#define PKV_DEV_BAD_BLOCK 2        /* block_table entry outside [0, num_blocks)      */
#define PKV_DEV_BAD_LENGTH 4       /* length > max_blocks_per_seq * block_size, < 0  */
#define PKV_DEV_TIMEOUT 8          /* a bounded wait inside a kernel gave up         */

#define PKV_BF16 0
#define PKV_F32 1

/* One-line reason for the last non-OK return on this thread ("" if none). */
const char* pkv_last_error(void);
/* Library ABI version (major * 100 + minor). */
int pkv_version(void);

/* ==========================================================================
 * Host-side block management (no device pointers)
 * ========================================================================== */

/* Opaque BlockPool: FIFO free queue plus a set that catches double frees
 * ("KV Cache 管理设计文档" §2.4). The queue starts as `initial_order` (a
 * permutation of 0..num_blocks-1; NULL = 0,1,2,...); the first id popped becomes
 * the null block, which is never handed out. Seeded shuffles are expressed by
 * passing a shuffled order. The pool is owned by the caller: destroy it with
 * pkv_pool_destroy. Not thread-safe. */
typedef struct pkv_pool pkv_pool;
int pkv_pool_create(int64_t num_blocks, const int32_t* initial_order, pkv_pool** out);
void pkv_pool_destroy(pkv_pool* pool);
int32_t pkv_pool_null_block(const pkv_pool* pool);
int64_t pkv_pool_num_free(const pkv_pool* pool);
/* Pop n ids from the head of the queue into ids_out[n]; all-or-nothing
 * (PKV_ERR_OUT_OF_BLOCKS leaves the pool unchanged). */
int pkv_pool_alloc(pkv_pool* pool, int64_t n, int32_t* ids_out);
/* Drop one reference per listed id; an id whose count reaches zero goes back to
 * the queue tail, in the listed order. PKV_ERR_DOUBLE_FREE (pool unchanged) if an
 * id is out of range, is the null block, or is listed more often than it is
 * referenced (an unshared block: free already, or listed twice). */
int pkv_pool_free(pkv_pool* pool, const int32_t* ids, int64_t n);
/* One more reference to each of ids[n], all currently held (a block shared by a
 * forked request, "KV Cache 笔记" fork_blocks). PKV_ERR_INVALID_ARG (pool
 * unchanged) if an id is free, out of range or the null block. */
int pkv_pool_share(pkv_pool* pool, const int32_t* ids, int64_t n);
/* Reference count of one block (0 = free or the null block; -1 = bad id). */
int32_t pkv_pool_ref_count(const pkv_pool* pool, int32_t id);

/* Skipped tokens of a manager after n computed tokens: 0 for full attention
 * (window <= 0), max(0, n - window + 1) for a sliding window
 * ("KV Cache 管理设计文档" §2.3 get_num_skipped_tokens). */
int64_t pkv_num_skipped_tokens(int64_t num_computed_tokens, int64_t window);

/* Batch block table [B, max_blocks_per_seq] (row-major, host memory) for sequences
 * of total length seq_lens[b] (including the newest token). Row b holds
 * ceil(len/bs) logical entries; with window > 0 the leading
 * floor(skipped(len - 1) / bs) entries, wholly outside the window, are the null
 * block and take nothing from the pool (§2.3.2); the others are popped from the
 * pool in FIFO order, sequence by sequence. Unused entries hold the null block.
 * All-or-nothing: PKV_ERR_OUT_OF_BLOCKS leaves the pool unchanged. */
int pkv_build_block_table(pkv_pool* pool, const int32_t* seq_lens, int32_t B, int32_t block_size,
                          int32_t window, int32_t max_blocks_per_seq, int32_t* table_out);
/* Static table arange(B * blocks_per_seq).reshape(B, -1) ("KVCache 优化技能" §3.2). */
int pkv_build_block_table_arange(int32_t B, int32_t blocks_per_seq, int32_t* table_out);
/* slot_mapping for num_new[b] tokens at positions start_pos[b].. of each sequence,
 * concatenated in sequence order (host memory). slot = table[b][pos / bs] * bs +
 * pos % bs ("KVCache 优化技能" §3.1; "KV Cache 管理设计文档" §4.2.2). Returns the
 * number of slots written (>= 0) or an error code. */
int64_t pkv_build_slot_mapping(const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* start_pos, const int32_t* num_new, int32_t B,
                               int32_t block_size, int32_t* slots_out, int64_t slots_capacity);

/* Pool sizing ("KV Cache 管理设计文档" §4.2.1 calculate_block_num); each "+1" is
 * the null block. */
int64_t pkv_block_num_fixed(int64_t max_concurrency, int64_t sliding_window, int64_t next_n,
                            int64_t block_size);
int64_t pkv_block_num_full_offline(int64_t max_len, int64_t block_size, int64_t max_concurrency);
int64_t pkv_block_num_full_online(int64_t available_bytes, int64_t per_token_bytes,
                                  int64_t block_size);

/* ==========================================================================
 * Request-level allocator ("KV Cache 管理设计文档" §2-§3; prefix sharing and
 * fork from "KV Cache 笔记", HF continuous batching). Host memory only.
 * ========================================================================== */

/* KVCacheManager over one manager per attention type (§2.2-§2.3). Type i has
 * window windows[i] (0 = full attention, > 0 = sliding window of that many
 * tokens), its own BlockPool of num_blocks[i] ids whose queue starts as
 * initial_orders[i] (NULL, or a NULL entry = 0,1,2,...), and group id i in block
 * fingerprints. At most one full-attention and one sliding-window type
 * (PKV_ERR_INVALID_ARG otherwise). prefix_caching != 0 turns on prefix sharing for
 * full-attention types. Owned by the caller (pkv_manager_destroy). Not
 * thread-safe. Request ids are any int64 values. */
typedef struct pkv_kv_manager pkv_kv_manager;
int pkv_manager_create(int32_t num_types, const int32_t* windows, const int64_t* num_blocks,
                       const int32_t* const* initial_orders, int32_t block_size,
                       int64_t max_model_len, int32_t prefix_caching, pkv_kv_manager** out);
void pkv_manager_destroy(pkv_kv_manager* mgr);

/* allocate_slots (§3): the request will hold K/V for positions
 * [0, min(computed + num_new + lookahead, max_model_len)). Phase 1, type by type:
 * give back the blocks of a sliding window that no query from position
 * min(computed, max_model_len) on can see (remove_skipped_blocks: they become the
 * null block), then count the new blocks the type needs; return 0 at the first
 * type whose pool cannot supply them, with nothing allocated. Phase 2: append the
 * new entries in every type (leading entries wholly before position
 * computed - W + 1 are the null block, the rest come from the pool in FIFO order).
 * Returns 1 (allocated), 0 (not enough blocks) or a negative error. */
int pkv_manager_allocate_slots(pkv_kv_manager* mgr, int64_t request_id, int64_t computed_tokens,
                               int64_t num_new_tokens, int64_t lookahead_tokens);
/* Logical block list of a request in type `type` (get_block_ids): writes up to
 * `capacity` ids and returns the list's length (0 for an unknown request). */
int64_t pkv_manager_get_block_ids(const pkv_kv_manager* mgr, int64_t request_id, int32_t type,
                                  int32_t* ids_out, int64_t capacity);
/* Release every block of the request in every type (free); unknown ids are a no-op. */
int pkv_manager_free(pkv_kv_manager* mgr, int64_t request_id);
int64_t pkv_manager_num_free(const pkv_kv_manager* mgr, int32_t type);
int32_t pkv_manager_null_block(const pkv_kv_manager* mgr, int32_t type);
int32_t pkv_manager_ref_count(const pkv_kv_manager* mgr, int32_t type, int32_t block);
/* format_usage: "full:used/total,sliding:used/total" in type order; used = blocks
 * handed out (the null block not counted), total = the pool's size. Writes a
 * NUL-terminated string (truncated to capacity) and returns its full length. */
int64_t pkv_manager_format_usage(const pkv_kv_manager* mgr, char* buf, int64_t capacity);
/* prepare_block_tables (§4.2.2) for type `type`: row b is request_ids[b]'s list,
 * padded with the null block, into table_out[B, max_blocks_per_seq].
 * PKV_ERR_INVALID_ARG if a list is longer than max_blocks_per_seq. */
int pkv_manager_block_table(const pkv_kv_manager* mgr, int32_t type, const int64_t* request_ids,
                            int32_t B, int32_t max_blocks_per_seq, int32_t* table_out);

/* Block fingerprint: BLAKE2b (RFC 7693) with an 8-byte digest, read little-endian,
 * over [parent_hash as 8 little-endian bytes, only when has_parent] + tokens as
 * int32 little-endian + group_id as int32 little-endian. The same in every process
 * (the pages' reason for not using a salted built-in hash). */
uint64_t pkv_block_hash(uint64_t parent_hash, int32_t has_parent, const int32_t* tokens,
                        int32_t num_tokens, int32_t group_id);
/* Prefix match for a new request (search_prefix_match): the longest run of
 * leading full blocks of tokens[num_tokens] whose fingerprint chain is held by a
 * live request in every type, never including the block of the last token, is
 * attached to request_id (one more reference per block). Returns the number of
 * cached tokens (a multiple of block_size; 0 with prefix caching off or a
 * sliding-window type present), or a negative error if request_id already holds
 * blocks. Follow with allocate_slots(request_id, cached, num_tokens - cached). */
int64_t pkv_manager_match_prefix(pkv_kv_manager* mgr, int64_t request_id, const int32_t* tokens,
                                 int64_t num_tokens);
/* Fingerprint the request's full blocks that are not fingerprinted yet, from its
 * tokens (call after their K/V is computed). A fingerprint already taken by
 * another block keeps that block. Fingerprints are forgotten when their block's
 * last reference is released. No-op without prefix caching. */
int pkv_manager_cache_blocks(pkv_kv_manager* mgr, int64_t request_id, const int32_t* tokens,
                             int64_t num_tokens);
/* fork_blocks: each of child_ids[num_children] (new requests) gets the first
 * ceil(num_tokens / block_size) entries of the parent's list. shareable != 0:
 * full blocks are shared (one more reference per child) and only an incomplete
 * last block is replaced by a new block to be copied; shareable == 0: every real
 * block is replaced by a new one to be copied. Null entries stay null. The copies
 * (source, destination) are written type by type, child by child, to
 * copy_src/copy_dst (capacity entries), and copies_per_type[num_types] gets each
 * type's count; run pkv_copy_blocks on every cache of a type with its pairs.
 * All-or-nothing: PKV_ERR_OUT_OF_BLOCKS or a too-small capacity
 * (PKV_ERR_INVALID_ARG) leaves everything unchanged. Returns the total copies. */
int64_t pkv_manager_fork(pkv_kv_manager* mgr, int64_t parent_id, const int64_t* child_ids,
                         int32_t num_children, int64_t num_tokens, int32_t shareable,
                         int32_t* copy_src, int32_t* copy_dst, int64_t capacity,
                         int64_t* copies_per_type);

/* ==========================================================================
 * Device calls
 * ========================================================================== */

/* Cache write through slot_mapping (standalone guide 模式二: the cache viewed as
 * [num_blocks * block_size, H_kv, d] takes row t at index slot_mapping[t]).
 *   k_cache [num_blocks, block_size, num_kv_heads, head_dim_k]  written
 *   v_cache [num_blocks, block_size, num_kv_heads, head_dim_v]  written; NULL
 *           (with v = NULL) writes the k side only
 *   k [num_tokens, num_kv_heads, head_dim_k], v [num_tokens, num_kv_heads, head_dim_v]
 *   slot_mapping [num_tokens] int32 (device)
 * The MLA latent write passes cache_nope as k (H_kv 1, 512) and cache_rope as v
 * (H_kv 1, 64). A bit-exact copy; slot < 0 skips the row; slot >= num_blocks *
 * block_size skips it and sets PKV_DEV_BAD_SLOT. Duplicate slots in one call are
 * undefined (one of the rows wins). Row sizes must be multiples of 16 bytes. With
 * num_tokens = 0 nothing is launched and k, v and slot_mapping may be NULL. */
int pkv_kv_cache_write(void* k_cache, void* v_cache, const void* k, const void* v,
                       const int32_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim_k,
                       int32_t head_dim_v, int* dev_status, void* stream);

/* Block copy for a fork ("KV Cache 笔记", fork_blocks: the incomplete last block
 * of a forked request is copied, full blocks are shared). cache is one device
 * cache tensor whose blocks are contiguous rows of block_bytes (any
 * [num_blocks, block_size, heads, dim] cache: block_bytes = block_size * heads *
 * dim * element size). For i in [0, n): block dst[i] becomes a bit copy of block
 * src[i]; src and dst are device int32 arrays. Sources must not be destinations of
 * the same call (pkv_manager_fork's pairs never are). A pair with an id outside
 * [0, num_blocks) is skipped and sets PKV_DEV_BAD_BLOCK. block_bytes must be a
 * positive multiple of 16 and cache 16-byte aligned (PKV_ERR_INVALID_ARG). */
int pkv_copy_blocks(void* cache, int64_t num_blocks, int64_t block_bytes, const int32_t* src,
                    const int32_t* dst, int64_t n, int* dev_status, void* stream);

/* Fused MLA cache write (standalone guide 模式三: the kv_a projection output goes
 * through kv_a_layernorm RMSNorm and RoPE and into nope_cache / rope_cache in one
 * step, optionally returning k_nope / k_rope). For each token t:
 *   k_nope[t] = bf16(x[0:512] / sqrt(mean(x[0:512]^2) + epsilon) * gamma)
 *   k_rope[t] = bf16(x[512:576] * cos[t] + rotate_half(x[512:576]) * sin[t]),
 *   rotate_half(r) = [-r[32:64], r[0:32]] (the Llama forward's RoPE, "KV Cache 笔记"),
 * with x = latent[t], arithmetic in fp32 and round-to-nearest-even results;
 * k_nope[t] goes to cache_nope row slot_mapping[t] and k_rope[t] to cache_rope.
 *   cache_nope [num_blocks, block_size, 1, 512] bf16, cache_rope [.., 1, 64] bf16
 *   k_nope_out [T, 512], k_rope_out [T, 64] bf16: optional copies (NULL = none)
 *   latent [T, 576] bf16 (512 latent + 64 rope), gamma [512] bf16
 *   cos, sin [T, 64] fp32 (per token, every rope element)
 *   slot_mapping [T] int32: negative skips the cache write of the row; a slot
 *   >= num_blocks * block_size is skipped and sets PKV_DEV_BAD_SLOT.
 * kv_lora_rank must be 512 and rope_dim 64 (PKV_ERR_UNSUPPORTED). All pointers
 * 16-byte aligned. Device pointers; asynchronous on `stream`. */
int pkv_mla_rmsnorm_rope_write(void* cache_nope, void* cache_rope, void* k_nope_out,
                               void* k_rope_out, const void* latent, const void* gamma,
                               const float* cos, const float* sin, const int32_t* slot_mapping,
                               int64_t num_tokens, int64_t num_blocks, int32_t block_size,
                               int32_t kv_lora_rank, int32_t rope_dim, float epsilon,
                               int* dev_status, void* stream);

/* Decode attention, one query token per sequence (sparse_mode 0 / band 4).
 * For each b, h: o = softmax(scale * q[b,h] . K^T) V over positions
 * [max(0, len_b - window), len_b) (window <= 0: [0, len_b)) of sequence b, read
 * through block_table; query head h uses kv head h / (H / H_kv) ("KV Cache 笔记",
 * MHA -> MQA -> GQA, repeat_kv). seq_lens counts every visible position including
 * the token just written (the FA reads up to the new token: skill note §3.6).
 *   out  [B, H, head_dim] (bf16 or fp32), lse [B, H] fp32 natural log (nullable);
 *        len_b = 0 gives o = 0, lse = -inf
 *   q    [B, H, head_dim] bf16
 *   k_cache, v_cache [num_blocks, block_size, H_kv, head_dim] bf16
 *   block_table [B, max_blocks_per_seq] int32; seq_lens [B] int32 (device)
 * Supported: head_dim 128, block_size 128, H % H_kv == 0, H / H_kv <= 16.
 * Entries of block_table outside the visible range are never read. */
size_t pkv_decode_workspace_size(int32_t B, int32_t H, int32_t H_kv, int32_t head_dim);

/* Kernel used by pkv_paged_attention_decode, process-wide (not thread-safe to change
 * while calls are in flight). PKV_KERNEL_AUTO picks the tcgen05 tensor-core kernel
 * for every group size; PKV_KERNEL_CUDA_CORE forces the CUDA-core kernel. Both
 * produce the same partial results up to fp32 rounding. */
#define PKV_KERNEL_AUTO 0
#define PKV_KERNEL_CUDA_CORE 1
#define PKV_KERNEL_TENSOR_CORE 2
int pkv_set_decode_kernel(int32_t kernel);
int32_t pkv_get_decode_kernel(void);
int pkv_paged_attention_decode(void* out, int32_t out_dtype, float* lse, const void* q,
                               const void* k_cache, const void* v_cache,
                               const int32_t* block_table, int32_t max_blocks_per_seq,
                               const int32_t* seq_lens, int32_t B, int32_t H, int32_t H_kv,
                               int32_t head_dim, int32_t block_size, int64_t num_blocks,
                               float scale, int32_t window, void* workspace,
                               size_t workspace_bytes, int* dev_status, void* stream);

/* Speculative (multi-token) decode: q_len new query rows per sequence, all already
 * written to the cache (MTP verification; standalone guide appendix C: a decode
 * step with q_len > 1 takes the prefill branch, sparse_mode 3, the bottom-right
 * causal mask; design doc: allocate_slots' lookahead_tokens reserve the slots of
 * the draft rows). Query row i of sequence b sits at position len_b - q_len + i
 * and, for each head h (kv head h / (H / H_kv)), attends to the keys at positions
 * p <= len_b - q_len + i, and with window > 0 only to p > len_b - q_len + i - window:
 * each row is the decode step of the prefix that ends at its own position. A row
 * whose position is negative (len_b < q_len) returns o = 0, lse = -inf. With a
 * window, block_table must keep the blocks from position len_b - q_len + 1 - window
 * on (the generator's window is window + q_len - 1).
 *   out [B, q_len, H, head_dim] (bf16 or fp32), lse [B, q_len, H] fp32 (nullable)
 *   q   [B, q_len, H, head_dim] bf16
 *   k_cache, v_cache [num_blocks, block_size, H_kv, head_dim] bf16
 *   block_table [B, max_blocks_per_seq] int32; seq_lens [B] int32 totals (device)
 * Supported: head_dim 128, block_size 128, q_len 1..4, q_len * H / H_kv <= 32
 * (PKV_ERR_UNSUPPORTED otherwise). q_len = 1 is pkv_paged_attention_decode.
 * Workspace: pkv_decode_spec_workspace_size(B, q_len, H, H_kv, head_dim) bytes,
 * 256-byte aligned. Device pointers; asynchronous on `stream`. */
size_t pkv_decode_spec_workspace_size(int32_t B, int32_t q_len, int32_t H, int32_t H_kv,
                                      int32_t head_dim);
int pkv_paged_attention_decode_spec(void* out, int32_t out_dtype, float* lse, const void* q,
                                    const void* k_cache, const void* v_cache,
                                    const int32_t* block_table, int32_t max_blocks_per_seq,
                                    const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H,
                                    int32_t H_kv, int32_t head_dim, int32_t block_size,
                                    int64_t num_blocks, float scale, int32_t window,
                                    void* workspace, size_t workspace_bytes, int* dev_status,
                                    void* stream);

/* Prefill attention over TND-packed queries (standalone guide: sparse_mode 3 for
 * TND paged prefill, q in cumulative form, kv in direct form; "KV Cache 笔记"
 * "手写40行": the causal mask is bottom-right aligned when a cache precedes the new
 * rows). Sequence b owns query rows [cu[b-1], cu[b]) (cu[-1] = 0), q_b rows, and
 * c_b = seq_lens_kv[b] - q_b cached positions before them; its new K/V rows must
 * already be in the cache (pkv_kv_cache_write). Query row r (0-based in the
 * sequence) of head h attends, with kv head h / (H / H_kv), to keys
 * j <= c_b + r when causal = 1, to all seq_lens_kv[b] keys when causal = 0.
 * q_len = 1 rows are decode rows and mix freely with prefill rows.
 *   out [num_tokens, H, head_dim] (bf16 or fp32), lse [num_tokens, H] fp32 (nullable)
 *   q [num_tokens, H, head_dim] bf16; cu_seqlens_q [B] int32 cumulative ends (no
 *   leading zero), seq_lens_kv [B] int32 direct totals, q_b <= seq_lens_kv[b]
 *   k_cache, v_cache [num_blocks, block_size, H_kv, head_dim] bf16
 * Supported: head_dim 128, block_size 128, H / H_kv in {1, 2, 4, 8, 16}.
 * Workspace: pkv_prefill_workspace_size() bytes (depends only on the device). */
size_t pkv_prefill_workspace_size(void);
int pkv_paged_attention_prefill(void* out, int32_t out_dtype, float* lse, const void* q,
                                const int32_t* cu_seqlens_q, int32_t num_tokens,
                                const void* k_cache, const void* v_cache,
                                const int32_t* block_table, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens_kv, int32_t B, int32_t H, int32_t H_kv,
                                int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                float scale, int32_t causal, void* workspace,
                                size_t workspace_bytes, int* dev_status, void* stream);

/* Absorbed MLA decode ("KVCache 优化技能" 模式三; standalone guide 模式三 FA absorb
 * call: key = value = cache_nope, query_rope / key_rope passed separately, one
 * latent kv head). For each b and query head h, over positions [0, len_b):
 *   s_j = scale * (q_nope[b,h] . nope_j + q_rope[b,h] . rope_j),  o = softmax(s) . nope
 *   out [B, H, kv_lora_rank] (bf16 or fp32), lse [B, H] fp32 natural log (nullable)
 *   q_nope [B, H, kv_lora_rank] bf16, q_rope [B, H, rope_dim] bf16
 *   cache_nope [num_blocks, block_size, 1, kv_lora_rank] bf16
 *   cache_rope [num_blocks, block_size, 1, rope_dim] bf16
 *   block_table [B, max_blocks_per_seq] int32, seq_lens [B] int32 (device)
 * New latent rows are written beforehand with pkv_kv_cache_write (k = nope,
 * v = rope). Supported: kv_lora_rank 512, rope_dim 64, block_size 128, H <= 128.
 * Workspace: pkv_mla_decode_workspace_size(B, H) bytes. */
size_t pkv_mla_decode_workspace_size(int32_t B, int32_t H);
int pkv_mla_paged_decode(void* out, int32_t out_dtype, float* lse, const void* q_nope,
                         const void* q_rope, const void* cache_nope, const void* cache_rope,
                         const int32_t* block_table, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, int32_t B, int32_t H, int32_t kv_lora_rank,
                         int32_t rope_dim, int32_t block_size, int64_t num_blocks, float scale,
                         void* workspace, size_t workspace_bytes, int* dev_status, void* stream);

/* Absorbed MLA decode of q_len new query rows per sequence (multi-token prediction
 * over an MLA cache: standalone guide appendix C, a decode step with q_len > 1 takes
 * sparse_mode 3, the bottom-right causal mask; scores as in pkv_mla_paged_decode).
 * All q_len new latent rows are already in the cache. Query row i of sequence b sits
 * at position len_b - q_len + i and attends to the positions p <= len_b - q_len + i;
 * a row whose position is negative (len_b < q_len) returns o = 0, lse = -inf.
 *   out [B, q_len, H, kv_lora_rank] (bf16 or fp32), lse [B, q_len, H] fp32 (nullable)
 *   q_nope [B, q_len, H, kv_lora_rank] bf16, q_rope [B, q_len, H, rope_dim] bf16
 *   caches, block_table as for pkv_mla_paged_decode; seq_lens [B] int32 totals
 * Supported: q_len 1..4 and the shapes of pkv_mla_paged_decode (PKV_ERR_UNSUPPORTED
 * otherwise); q_len = 1 is pkv_mla_paged_decode. Each row is its own problem: the
 * rows of one sequence run on different CTA pairs at the same time, so their reads
 * of a latent tile meet in L2 rather than each coming from HBM.
 * Workspace: pkv_mla_decode_spec_workspace_size(B, q_len, H) bytes, 256-byte
 * aligned. Device pointers; asynchronous on `stream`. */
size_t pkv_mla_decode_spec_workspace_size(int32_t B, int32_t q_len, int32_t H);
int pkv_mla_paged_decode_spec(void* out, int32_t out_dtype, float* lse, const void* q_nope,
                              const void* q_rope, const void* cache_nope, const void* cache_rope,
                              const int32_t* block_table, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens, int32_t B, int32_t q_len, int32_t H,
                              int32_t kv_lora_rank, int32_t rope_dim, int32_t block_size,
                              int64_t num_blocks, float scale, void* workspace,
                              size_t workspace_bytes, int* dev_status, void* stream);

/* FP8 (E4M3) KV cache: write and decode. A quantised cache halves the bytes a decode
 * step reads. The pages list KV quantisation (skill note 高阶特性: INT8 / W8A8C8;
 * "KV Cache 笔记": KIVI-style grouped quantisation) and warn that dequantising into
 * temporary tensors every step eats the saving; here the decode kernel widens the
 * codes on chip and nothing is materialised.
 * Format: one fp32 scale per (token, kv head) row of head_dim values,
 * scale = amax / 448 (IEEE fp32 division), code = E4M3(x / scale) rounded to nearest
 * even with saturation to +-448 (the "fn" variant: no infinities, S.1111.111 =
 * NaN); an all-zero row has scale 0 and zero codes. value = code * scale.
 *   k_cache, v_cache [num_blocks, block_size, H_kv, head_dim] uint8 codes
 *   k_scale, v_scale [num_blocks, H_kv, block_size] fp32 (a block's scales of one
 *                    kv head are contiguous)
 * head_dim must be 128 (PKV_ERR_UNSUPPORTED). */

/* Quantise new rows k, v [num_tokens, H_kv, head_dim] bf16 and write codes and
 * scales through slot_mapping (negative slot: skipped; slot >= num_blocks *
 * block_size: skipped and PKV_DEV_BAD_SLOT). Caches 16-byte aligned, scales 4. */
int pkv_kv_cache_write_fp8(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                           const void* k, const void* v, const int32_t* slot_mapping,
                           int64_t num_tokens, int64_t num_blocks, int32_t block_size,
                           int32_t num_kv_heads, int32_t head_dim, int* dev_status, void* stream);
/* pkv_paged_attention_decode over an FP8 cache: same arguments, result, workspace
 * (pkv_decode_workspace_size) and error behaviour, plus the two scale arrays
 * (16-byte aligned). The attention is that of the dequantised cache; q stays bf16.
 * Rows of positions outside [max(0, len - window), len) are never used, whatever
 * bytes they hold. Always runs on the tensor cores. */
int pkv_paged_attention_decode_fp8(void* out, int32_t out_dtype, float* lse, const void* q,
                                   const void* k_cache, const void* v_cache, const float* k_scale,
                                   const float* v_scale, const int32_t* block_table,
                                   int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t B,
                                   int32_t H, int32_t H_kv, int32_t head_dim, int32_t block_size,
                                   int64_t num_blocks, float scale, int32_t window,
                                   void* workspace, size_t workspace_bytes, int* dev_status,
                                   void* stream);

/* Decode without any caller-provided scratch. The paper has no counterpart for
 * this call; it exists for callers that cannot allocate device memory (a plugin
 * inside a runtime that owns the allocator, a serving loop whose HBM is already
 * fully partitioned, code that must not risk the device synchronisation a
 * cudaMalloc can cause). Same arguments and result as pkv_paged_attention_decode
 * minus the workspace: the split-KV partials live in a file-scope device array of
 * PKV_DECODE_STATIC_SCRATCH_BYTES that every GPU loading the library keeps until
 * the process exits.
 *   - Rejects (PKV_ERR_WORKSPACE) any problem whose workspace would exceed that
 *     size (pkv_decode_workspace_size(B, H, H_kv, head_dim) tells).
 *   - Allocates nothing and calls no allocating routine.
 *   - The first call on a device, with that device current, looks up the array's
 *     device address (cudaGetSymbolAddress) and caches it for the process; make
 *     that first call before any stream capture. The cached address belongs to the
 *     device's primary context: it is not valid across cudaDeviceReset or in a
 *     non-primary driver context.
 *   - Runs on the current device, with its copy of the array: the pointers and
 *     `stream` must belong to that device.
 *   - All calls share the one array, which keeps the last call's contents. No part
 *     of it needs to start at zero. Calls that overlap on the GPU (other streams,
 *     other host threads) race on it: serialise them. */
#define PKV_DECODE_STATIC_SCRATCH_BYTES (8 * 1024 * 1024)
int pkv_paged_attention_decode_static(void* out, int32_t out_dtype, float* lse, const void* q,
                                      const void* k_cache, const void* v_cache,
                                      const int32_t* block_table, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t B, int32_t H, int32_t H_kv,
                                      int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                      float scale, int32_t window, int* dev_status, void* stream);

/* ==========================================================================
 * Self-test (no counterpart in the pages: a check of the kernels' failure path)
 * ========================================================================== */

/* Launches one small kernel that waits, with the bounded wait routines every
 * attention kernel uses, on an mbarrier that nothing completes. Each wait gives up
 * after its cycle limit (about a second at full clock) and the kernel sets
 * PKV_DEV_TIMEOUT in *dev_status (device memory, caller-owned; other bits are left
 * as they are), then returns: the CUDA context stays usable. Asynchronous on
 * `stream`. Errors: PKV_ERR_INVALID_ARG for a null dev_status; PKV_ERR_LAUNCH if
 * the launch fails. */
int pkv_selftest_bounded_wait(int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PAGED_KV_H */
