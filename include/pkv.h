/*
 * pkv.h — C ABI of the GB300 (sm_103a) paged-KV attention step for Qwen3-style
 * attention: per-head q/k RMSNorm, RoPE (theta = 1e6), the slot_mapping
 * scatter into a paged KV cache of 256-token blocks, and causal GQA attention
 * (32 query heads over 8 KV heads, head_dim 128) read through per-sequence
 * block tables, for single-token decode and for varlen prefill.
 *
 * Sources of the operations:
 *   "Nano-vLLM深度解读（下）" — §2 (Qwen3Attention: q_norm/k_norm, rotary_emb,
 *      attn), §4 (attention.py: store_kvcache_kernel, Attention.forward).
 *   "同一个 Qwen3，两种写法：从 transformers 到 nano-vllm 的推理改造" — §2 (the
 *      Qwen3-8B config), §3.2 (flat varlen layout, cu_seqlens), §3.3 (paged
 *      cache, slot = block_id * block_size + offset), §3.4 (the two attention
 *      entry points, GQA, "store first, then read"), §3.5 (RoPE table),
 *      §3.6 (RMSNorm rounding points).
 *
 * Conventions shared by every call
 *   - bf16 tensors are passed as void* to bf16 data (2-byte elements), int
 *     tensors as int32_t*.  All tensor pointers are DEVICE pointers on the
 *     current CUDA device and must be 16-byte aligned; rows are contiguous.
 *   - Fixed geometry: 32 query heads, 8 KV heads, head_dim 128, block_size
 *     256, positions < 40960.  A cache is bf16 [num_blocks, 256, 8, 128]:
 *     token row `slot` starts at element slot * 1024, head h of it at
 *     slot * 1024 + h * 128.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work: they never synchronise, and results are ready when the
 *     stream reaches that point.  No call allocates device memory except the
 *     first call on a device (or pkv_init), which uploads the 20 MiB fp32
 *     RoPE table and a 4-byte error word for that device.
 *   - The caller owns every tensor and workspace; the library keeps only the
 *     per-device RoPE table and error word until pkv_shutdown().
 *   - Return value: PKV_OK (0) or a negative pkv_status.  On error nothing
 *     is enqueued and pkv_last_error() (thread-local) says why.  Host-side
 *     checks cover null pointers, sizes, alignment and strides.  A call with
 *     nothing to do (no tokens, no sequences or no queries) returns PKV_OK
 *     once its sizes are known not to be negative, before any pointer is
 *     read, so empty tensors may have NULL data.  Checks that
 *     need device data (a position >= 40960, a slot outside the cache, a
 *     block id outside [0, num_blocks), a context longer than its block-table
 *     row) are made inside the kernels: the offending token / sequence is
 *     skipped (its outputs are left unwritten or zero, as each call says) and
 *     a bit is set in the device's error word, which pkv_check_errors()
 *     reads.  Kernels never trap; every wait inside them is bounded.
 *   - Debug mode: with PKV_DEBUG set to anything but "0" in the environment
 *     (read once per process), every compute call synchronises its stream
 *     after the launch and returns PKV_ERR_CUDA if the kernel faulted or
 *     PKV_ERR_BOUNDS if it set an error bit.  The bits are read and cleared as
 *     pkv_check_errors() does; for pkv_attn_decode_noalloc, only its own
 *     word, and a caller's error word is left to the caller.  A call on a
 *     stream that is being captured into a CUDA graph is not checked.  The
 *     outputs are the same as without the mode; only the call returns later.
 *   - Thread safety: calls may come from several host threads; calls that
 *     write the same tensors must be ordered by the caller.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_NUM_Q_HEADS 32
#define PKV_NUM_KV_HEADS 8
#define PKV_HEAD_DIM 128
#define PKV_BLOCK_SIZE 256
#define PKV_MAX_POSITION 40960
#define PKV_ROPE_THETA 1.0e6
#define PKV_RMS_EPS 1.0e-6f
#define PKV_HIDDEN 4096 /* Qwen3-8B hidden size: rows of the decoder layer's RMSNorm */
#define PKV_QKV_OUT 6144 /* output features of the fused QKV projection: 32*128 + 2 * 8*128 */

typedef enum pkv_status {
  PKV_OK = 0,
  PKV_ERR_NULL = -1,        /* a required pointer is NULL */
  PKV_ERR_SHAPE = -2,       /* a size or stride is negative, zero where it must not be, or inconsistent */
  PKV_ERR_UNSUPPORTED = -3, /* a request outside the fixed geometry */
  PKV_ERR_BOUNDS = -4,      /* returned by pkv_check_errors when a kernel met an out-of-range index */
  PKV_ERR_CUDA = -5,        /* a CUDA runtime / driver call failed (the message names it) */
  PKV_ERR_NO_DEVICE = -6,   /* no CUDA device, or the device is not sm_103 */
  PKV_ERR_ALIGN = -7,       /* a pointer or row stride is not 16-byte aligned */
  PKV_ERR_WORKSPACE = -8    /* the workspace is missing or smaller than required */
} pkv_status;

/* Device error-word bits (see pkv_check_errors). */
#define PKV_EFLAG_POSITION 0x1u /* a position outside [0, 40960): token skipped */
#define PKV_EFLAG_SLOT 0x2u     /* a slot outside [-1, num_blocks*256): K/V of that token not stored */
#define PKV_EFLAG_BLOCK_ID 0x4u /* a block id outside [0, num_blocks): its keys were treated as absent */
#define PKV_EFLAG_CONTEXT 0x8u  /* a context / key length beyond the block-table row, max_context or max_seqlen */
#define PKV_EFLAG_TIMEOUT 0x10u /* a bounded wait inside a kernel gave up: results of that call are invalid */
#define PKV_EFLAG_SEQLEN 0x20u  /* a prefill sequence with more queries than keys: its rows were zeroed */

/* Message for the last failing call on this host thread ("" if none). */
const char* pkv_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

/* Optional eager set-up for `device` (uploads the RoPE table, allocates the
 * error word).  Without it the first call on a device does this lazily; call
 * it before capturing calls into a CUDA graph. */
int pkv_init(int device);

/* Free the per-device state of every device.  No call may be in flight. */
int pkv_shutdown(void);

/* Synchronise `stream`, then read and clear the current device's error word
 * into *flags (may be NULL).  Returns PKV_ERR_BOUNDS if any bit was set,
 * PKV_OK otherwise. */
int pkv_check_errors(void* stream, uint32_t* flags);

/*
 * pkv_qknorm_rope_store — steps a1..a3 of one layer, fused in one kernel.
 *
 * For every token t < num_tokens, in the order Qwen3Attention.forward uses
 * ("Nano-vLLM深度解读（下）" §2):
 *   1. q_norm / k_norm: RMSNorm over head_dim of each of the 32 q heads and
 *      8 k heads, eps 1e-6, fp32 arithmetic; the normalised value is rounded
 *      to bf16, multiplied by the bf16 weight and rounded to bf16
 *      ("同一个 Qwen3，两种写法" §3.6).
 *   2. RoPE at positions[t], theta 1e6, half split: y1 = x1 cos - x2 sin,
 *      y2 = x2 cos + x1 sin in fp32 from an fp32 cos/sin table, rounded to
 *      bf16 once (same page, §3.5).
 *   3. The store of "Nano-vLLM深度解读（下）" §4: if slot_mapping[t] != -1,
 *      the normalised+rotated k row (8 heads) and the v row are copied to
 *      row slot_mapping[t] of k_cache / v_cache.
 *
 *   q            bf16 [num_tokens, 32, 128], row stride q_row_stride elements;
 *                rewritten IN PLACE with the normalised, rotated q.
 *   k, v         bf16 [num_tokens, 8, 128], row strides k_row_stride /
 *                v_row_stride (elements); read only.  (q, k, v may be views
 *                of one fused [T, 6144] qkv buffer.)
 *   positions    int32 [num_tokens], each in [0, 40960).
 *   slot_mapping int32 [num_tokens], -1 (do not store) or in [0, num_blocks*256).
 *   q_norm_w, k_norm_w  bf16 [128].
 *   k_cache, v_cache    bf16 [num_blocks, 256, 8, 128]; written only at mapped rows.
 * Row strides must be multiples of 8 elements and at least 4096 (q) / 1024
 * (k, v).  num_tokens == 0 is a no-op (see above).  Different tokens must not map to the
 * same slot (the winner would be unspecified).
 */
int pkv_qknorm_rope_store(void* q, int64_t q_row_stride, const void* k, int64_t k_row_stride, const void* v,
                          int64_t v_row_stride, const int32_t* positions, const int32_t* slot_mapping,
                          const void* q_norm_w, const void* k_norm_w, void* k_cache, void* v_cache,
                          int64_t num_tokens, int64_t num_blocks, void* stream);

/*
 * Workspace bytes pkv_attn_decode needs for `batch` sequences whose context
 * lengths are at most `max_context` (0 if the call will split no sequence).
 */
size_t pkv_attn_decode_workspace_size(int32_t batch, int32_t max_context);

/*
 * pkv_attn_decode — step a4: paged GQA attention of one query token per
 * sequence over its cached keys ("Nano-vLLM深度解读（下）" §4, decode branch:
 * flash_attn_with_kvcache with cache_seqlens = context_lens and a block
 * table; "同一个 Qwen3，两种写法" §3.4).
 *
 * For sequence b and query head h, with L = context_lens[b] and g = h / 4:
 *   out[b, h] = sum_j softmax_j(scale * q[b, h] . K_j) V_j  over j < L,
 * where K_j / V_j are head g of cache row block_table[b, j / 256] * 256 +
 * j % 256.  context_lens includes the token stored by this step (the store
 * runs first).  Split-K: a sequence's keys are cut into chunks processed by
 * separate CTAs and merged by log-sum-exp in fp32.
 *
 *   q            bf16 [batch, 32, 128] (contiguous).
 *   k_cache, v_cache  bf16 [num_blocks, 256, 8, 128].
 *   context_lens int32 [batch], 0 <= L <= min(max_context, max_blocks_per_seq * 256).
 *                L == 0 gives a zero output row.
 *   block_table  int32 [batch, max_blocks_per_seq]; only the first
 *                ceil(L / 256) entries of row b are read (others may hold -1).
 *   max_context  host-side upper bound of context_lens (sizes the split).
 *   scale        softmax scale (1/sqrt(128) for Qwen3).
 *   out          bf16 [batch, 32, 128].
 *   workspace    device memory of at least pkv_attn_decode_workspace_size(batch,
 *                max_context) bytes, 256-byte aligned, ZERO-FILLED BEFORE ITS
 *                FIRST USE; every call leaves its counters at zero again.  May
 *                be NULL when that size is 0.  Calls sharing a workspace must
 *                not overlap on the GPU.
 */
int pkv_attn_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* context_lens,
                    const int32_t* block_table, int32_t batch, int32_t max_blocks_per_seq, int64_t num_blocks,
                    int32_t max_context, float scale, void* out, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * pkv_attn_decode_noalloc — pkv_attn_decode for callers that cannot allocate
 * device memory (a sealed memory pool, an allocator-free embedding, a process
 * that hands out all of its device memory up front).  The pages have no
 * counterpart to this entry point; it exists for those callers only.
 *
 * Same operation, arguments and results as pkv_attn_decode, but no workspace
 * is passed: the split-K scratch is a static array of 8 MiB inside the
 * library, held by every GPU that loads the library until the process exits.
 * The call never allocates (no cudaMalloc, cudaFree or allocating library
 * routine).  Its first call on a device, with that device current, looks up
 * the array's device address (cudaGetSymbolAddress) and sets the kernel's
 * shared-memory limit; make that first call before any stream capture.
 * Every call shares the array and it keeps the last call's contents: the
 * call clears the split counters it needs before its kernel runs, and calls
 * that overlap on the GPU (other streams, other threads) race on the array.
 * A (batch, max_context) whose split scratch would exceed 8 MiB is rejected
 * with PKV_ERR_WORKSPACE (splits are only used for batch < 76, which always
 * fits; the check is there for completeness).
 *
 *   error_flags  optional device pointer to a uint32 the kernel ORs the
 *                PKV_EFLAG_* bits into.  With NULL the bits go to a word in
 *                static device memory, which pkv_check_errors reads and clears
 *                with the library's own error word (pkv_check_errors sets up
 *                the library's per-device state, an allocation, on its first
 *                call: a caller that cannot allocate at all passes its own
 *                error_flags word and reads it itself).
 */
int pkv_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache, const int32_t* context_lens,
                            const int32_t* block_table, int32_t batch, int32_t max_blocks_per_seq,
                            int64_t num_blocks, int32_t max_context, float scale, void* out, uint32_t* error_flags,
                            void* stream);

/*
 * pkv_attn_prefill — step a5: causal varlen attention of a flat batch of
 * query tokens over the paged cache ("Nano-vLLM深度解读（下）" §4, prefill
 * branch with a block table: flash_attn_varlen_func(q, k_cache, v_cache,
 * cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, causal=True,
 * block_table); "同一个 Qwen3，两种写法" §3.2 and §3.4).
 *
 * Sequence s owns query rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 (Lq rows)
 * and keys 0 .. Lk-1 with Lk = cu_seqlens_k[s+1] - cu_seqlens_k[s], read
 * through block_table row s.  Query row i sits at position Lk - Lq + i and
 * sees keys 0 .. Lk - Lq + i (causal, aligned to the end of the keys, which
 * covers prefix-cached and chunked prefill).  GQA: q head h reads KV head h/4.
 * Keys are always read from the cache, so pkv_qknorm_rope_store must have
 * stored this step's tokens first.
 *
 *   q            bf16 [total_q, 32, 128] (contiguous), total_q = cu_seqlens_q[num_seqs].
 *   cu_seqlens_q, cu_seqlens_k  int32 [num_seqs + 1], non-decreasing, from 0.
 *   block_table  int32 [num_seqs, max_blocks_per_seq].
 *   max_seqlen_q, max_seqlen_k  host-side upper bounds of Lq and Lk.
 *   out          bf16 [total_q, 32, 128].  Rows of a sequence with Lq > Lk
 *                are zeroed (PKV_EFLAG_SEQLEN); so are the rows of a sequence
 *                whose Lk exceeds its table row or the max_seqlen bounds
 *                (PKV_EFLAG_CONTEXT).  A block id outside [0, num_blocks)
 *                contributes no keys (PKV_EFLAG_BLOCK_ID), as in decode.
 */
int pkv_attn_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* cu_seqlens_q,
                     const int32_t* cu_seqlens_k, const int32_t* block_table, int32_t num_seqs,
                     int32_t max_blocks_per_seq, int64_t num_blocks, int32_t total_q, int32_t max_seqlen_q,
                     int32_t max_seqlen_k, float scale, void* out, void* stream);

/*
 * pkv_add_rmsnorm — the decoder layer's RMSNorm with the pending residual add
 * folded in ("同一个 Qwen3，两种写法" §3.6, nano-vllm add_rms_forward; the
 * step that feeds the QKV projection of this attention step).
 *
 * For each token t (rows of PKV_HIDDEN = 4096 bf16 elements, contiguous):
 *   s = fp32(x[t]) + fp32(residual[t]);  residual[t] <- bf16(s);
 *   out[t] = bf16(bf16(s * rsqrt(mean(s*s) + eps)) * weight)
 * The mean is over the unrounded fp32 sum.  With residual == NULL (the first
 * layer) s = fp32(x[t]) and nothing else is written: the caller keeps x as
 * the residual.  HBM traffic: 4 rows per token (3 without residual).
 *
 *   x         bf16 [num_tokens, 4096], read only (out may equal x: in place).
 *   residual  bf16 [num_tokens, 4096], read and overwritten; NULL for none.
 *             Must not alias x or out.
 *   weight    bf16 [4096].
 *   out       bf16 [num_tokens, 4096].
 *   hidden    must be PKV_HIDDEN (else PKV_ERR_UNSUPPORTED).
 *   eps       >= 0 (Qwen3: PKV_RMS_EPS).
 * All pointers 16-byte aligned.  Asynchronous on `stream`.
 */
int pkv_add_rmsnorm(const void* x, void* residual, const void* weight, void* out, int64_t num_tokens,
                    int32_t hidden, float eps, void* stream);

/*
 * pkv_qkv_rope_store — the QKV projection with pkv_qknorm_rope_store's work
 * as its epilogue ("同一个 Qwen3，两种写法" §3.1: one GEMM for q, k and v with
 * their weights concatenated along the output dimension, then the split;
 * "Nano-vLLM深度解读（下）" §2 Qwen3Attention.forward: q_norm/k_norm, rotary
 * embedding; §4 store_kvcache).
 *
 *   y = bf16(x W^T): x bf16 [T, 4096] (row-major), w_qkv bf16 [6144, 4096]
 *   (rows 0..4095 the q heads, 4096..5119 the k heads, 5120..6143 the v heads,
 *   128 rows per head, as nn.Linear stores a weight), fp32 accumulation.
 *   q_out bf16 [T, 32, 128] <- norm + RoPE of the q part (positions as in
 *   pkv_qknorm_rope_store); k_cache / v_cache rows at slot_mapping[t] <- the
 *   normed + rotated k part and the raw v part (slot -1: not stored).  The
 *   norm, rounding points, RoPE table and error flags are those of
 *   pkv_qknorm_rope_store, applied to the bf16 projection.
 * All pointers 16-byte aligned (index arrays 4-byte).  Asynchronous.
 */
int pkv_qkv_rope_store(const void* x, const void* w_qkv, const int32_t* positions, const int32_t* slot_mapping,
                       const void* q_norm_w, const void* k_norm_w, void* q_out, void* k_cache, void* v_cache,
                       int64_t num_tokens, int64_t num_blocks, void* stream);

/* ------------------------------------------------------------------------
 * Block manager (host only, no GPU): the control plane that produces the
 * block_table rows and slot_mapping entries the calls above consume
 * ("Nano-vLLM深度解读（下）" §4, the CPU-side Block Manager: sequences,
 * block allocation, reference counts, prefix-cache reuse; "同一个 Qwen3，两种
 * 写法" §3.3: slot = physical block * 256 + offset, blocks shared by
 * sequences with the same prefix are stored once).
 *
 * A pool of num_blocks blocks of PKV_BLOCK_SIZE tokens.  Full blocks carry a
 * hash chained over the prefix (FNV-1a 64-bit of the previous block's hash
 * and the block's token ids; a lookup also compares the ids).  Allocating a
 * prompt reuses the longest run of leading full blocks already in the pool
 * (their tokens are "cached": no new KV) and takes free blocks for the rest.
 * A block whose reference count drops to 0 goes to the back of the free list
 * with its contents and hash, and can still be reused until it is handed
 * out again.  Functions return PKV_OK or a negative PKV_ERR_* code with a
 * message in pkv_last_error(); on an error nothing is changed.  One manager
 * must not be used from several threads at once.
 * ------------------------------------------------------------------------ */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager over blocks 0..num_blocks-1 (all free).  NULL on error. */
pkv_block_manager* pkv_bm_create(int32_t num_blocks);
void pkv_bm_destroy(pkv_block_manager* bm);
/* Free blocks (reference count 0), or -1 for a NULL manager. */
int64_t pkv_bm_num_free_blocks(const pkv_block_manager* bm);
/* Reference count of one block (number of sequences holding it), or -1. */
int32_t pkv_bm_ref_count(const pkv_block_manager* bm, int32_t block);
/* Blocks for a prompt of num_tokens >= 1 token ids (host array).  Needs
 * ceil(num_tokens/256) free blocks (PKV_ERR_WORKSPACE otherwise).
 * *num_cached_tokens (may be NULL) receives the number of leading tokens
 * whose blocks were reused: their KV is in the cache already. */
int pkv_bm_allocate(pkv_block_manager* bm, int64_t seq_id, const int32_t* token_ids, int32_t num_tokens,
                    int32_t* num_cached_tokens);
/* One more token for an allocated sequence (decode): a token that starts a
 * block takes a free block, a token that fills one gives it its hash.
 * *slot (may be NULL) receives the cache row of the new token. */
int pkv_bm_append(pkv_block_manager* bm, int64_t seq_id, int32_t token_id, int32_t* slot);
/* Release a sequence's blocks (reference counts drop, last block first). */
int pkv_bm_free(pkv_block_manager* bm, int64_t seq_id);
/* Length, block count and cached-prefix length of a sequence (NULLs allowed). */
int pkv_bm_seq_info(const pkv_block_manager* bm, int64_t seq_id, int32_t* num_tokens, int32_t* num_blocks,
                    int32_t* num_cached_tokens);
/* block_table rows for num_seqs sequences: int32 [num_seqs, max_blocks] (host),
 * padded with -1; PKV_ERR_SHAPE if a sequence holds more than max_blocks. */
int pkv_bm_block_table(const pkv_block_manager* bm, const int64_t* seq_ids, int32_t num_seqs, int32_t* table,
                       int32_t max_blocks);
/* Cache rows of token positions [start, end) of one sequence (host int32). */
int pkv_bm_slot_mapping(const pkv_block_manager* bm, int64_t seq_id, int32_t start, int32_t end, int32_t* slots);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
