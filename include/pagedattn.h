/*
 * pagedattn.h -- C ABI of the GB300 (sm_103a) paged KV-cache attention library
 * (libpagedattn.so).
 *
 * What it computes: O = softmax(scale * Q K^T) V per query head, optionally
 * causal (bottom-right aligned: query row i of Lq sees keys t <= i + Lk - Lq),
 * for MHA and GQA (query head h reads kv head h / (Hq/Hkv)).  K and V are read
 * through a per-sequence block table of pages of 16 to 256 tokens (or from a
 * contiguous cache), with per-sequence lengths taken from device arrays -- the flash_attn_with_kvcache /
 * flash_attn_varlen_func interface discussed on
 *   flash-attention #824 "Add support for small page sizes" (reproduction
 *     snippet; page size 16; k=/v= append through block_table),
 *   vLLM #6052 "Unify the kernel used in flash attention backend" (one varlen
 *     launch for prefill and decode; CUDA-graph padding rules),
 *   flash-attention #1000 "Inappropriate Number of Splits Predicted by
 *     determine_num_splits" (split-KV on a preallocated contiguous cache;
 *     cache_seqlens lives on the GPU and must not be read by the host),
 *   vLLM #3010 "Introduce flash-attn (>= 2.5.0)" (paged decode and
 *     prefill-with-cache-write benchmarks, MHA and GQA).
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers owned by the caller, except where a
 *     comment says otherwise.  The library allocates nothing and never
 *     synchronises; every call is ordered on `stream` (a cudaStream_t; 0 is
 *     the legacy default stream) and reads lengths only on the GPU.
 *   - Element types: PA_F16 or PA_BF16; q, caches, new k/v and out share it.
 *     Softmax statistics, partial outputs and LSE are fp32.  LSE is the
 *     natural-log log-sum-exp of the scaled scores; rows with no visible key
 *     produce O = 0 and LSE = -inf.
 *   - head_dim D must be 64 or 128; a paged cache's page size is 16, 32, 64,
 *     128 or 256 tokens (page_size argument); Hq must be a multiple of Hkv.
 *   - Cache tensors are described by pa_tensor4 (element strides; the D axis
 *     is contiguous).  Base pointers must be 16-byte aligned and all three
 *     strides multiples of 8 elements (16 bytes), because K/V tiles are
 *     fetched with the Tensor Memory Accelerator.
 *   - Return value: PA_OK (0) or a negative PA_ERR_* code for a rejected
 *     argument or a failed launch.  Errors the GPU finds while running
 *     (block-table entries outside the pool, lengths beyond the table or the
 *     cache, a pipeline wait that timed out) are written to `err_word`
 *     (int32[4] in device memory, zeroed by the caller; may be NULL):
 *     err_word[0] = first PA_DEVERR_* code, [1] = sequence index, [2] = the
 *     offending value.  The kernels never fault on such input: an out-of-range
 *     page is replaced by page 0 for reading and is never written.
 *   - pa_last_error_string() describes the last non-OK return on the calling
 *     thread.
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

typedef struct CUstream_st* pa_stream_t; /* same type as cudaStream_t */

enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad stride or alignment */
  PA_ERR_UNSUPPORTED = -2, /* dtype, head_dim, Hq % Hkv, or shape outside the kernels */
  PA_ERR_CUDA = -3,        /* a CUDA runtime call or kernel launch failed */
  PA_ERR_WORKSPACE = -4    /* workspace pointer NULL or smaller than required */
};

enum { PA_F16 = 0, PA_BF16 = 1 };

/* Codes written to err_word[0] by the kernels. */
enum {
  PA_DEVERR_PAGE_OOB = 1,    /* block_table entry < 0 or >= num_pages            */
  PA_DEVERR_LENGTH = 2,      /* length < 0, beyond the table, cache or max_seqlen_k */
  PA_DEVERR_TIMEOUT = 3      /* a pipeline wait exceeded its time limit          */
};

/* A 4-D cache view.  Paged: [num_pages, page_size, Hkv, D] with stride_b =
 * elements between pages, stride_t between the token slots of a page,
 * stride_h between kv heads.  Contiguous (block_table == NULL):
 * [B, capacity, Hkv, D] with stride_b between sequences.
 *
 * page_size (the paged calls' argument): tokens per page, one of 16, 32, 64,
 * 128, 256 -- vLLM's 16-token blocks and the 256-token pages flash-attention
 * required, which vLLM #3010 "Introduce flash-attn" compares (cache-write cost
 * at context 512 / 1024).  Ignored when block_table == NULL; any other value
 * with a block table returns PA_ERR_UNSUPPORTED.  Position pos of sequence b
 * is in page block_table[b * bt_stride + pos / page_size], slot
 * pos % page_size. */
typedef struct {
  void* ptr;
  int64_t stride_b;
  int64_t stride_t;
  int64_t stride_h;
} pa_tensor4;

/*
 * pa_append_kv -- write new tokens' k/v into the cache (a bit copy).
 *
 * For every b < B, i < Lnew, kv head g: position pos = cache_seqlens[b] + i
 * receives k_new[b, i, g, :] (and v_new likewise) at page
 * block_table[b * bt_stride + pos / page_size], slot pos % page_size; or, with
 * block_table == NULL, at row [b, pos] of a contiguous cache.  The k=/v=
 * append of flash_attn_with_kvcache (flash-attention #824, reproduction
 * snippet and the reply noting that the call allocates nothing and writes
 * through block_table).  cache_seqlens is input only and is not updated.
 *
 *   k_new, v_new  [B, Lnew, Hkv, D] contiguous.
 *   block_table   int32 [B, >= max_pages] rows of stride bt_stride, or NULL.
 *   cache_extent  paged: number of pages in the pool; contiguous: capacity
 *                 (tokens) of each sequence.
 * Positions outside the table (pos / page_size >= max_pages) or the capacity, and
 * out-of-pool pages, are skipped and reported in err_word.  Appends of two
 * sequences that share a physical page race (the caller's responsibility).
 */
PA_API int pa_append_kv(pa_tensor4 k_cache, pa_tensor4 v_cache, const void* k_new,
                        const void* v_new, const int32_t* cache_seqlens,
                        const int32_t* block_table, int64_t bt_stride, int max_pages,
                        int page_size, int B, int Lnew, int Hkv, int D, int64_t cache_extent,
                        int dtype, int32_t* err_word, pa_stream_t stream);

/*
 * pa_fwd_kvcache -- flash_attn_with_kvcache forward: decode, multi-query
 * decode and causal prefill over a paged (or contiguous) cache, with optional
 * in-kernel append and split-KV.
 *
 * Sequence b attends over Lk_b = cache_seqlens[b] + Lnew keys: positions
 * below cache_seqlens[b] come from the cache, positions at or above it are
 * the Lnew new tokens, which are also written into the cache (as
 * pa_append_kv) in the same call.  (flash-attention #824: reproduction
 * snippet; flash-attention #1000: split-KV and the host-side num_splits
 * problem; vLLM #3010: paged decode table.)
 *
 *   q            [B, Lq, Hq, D], element strides q_sb, q_st, q_sh (multiples
 *                of 8); D contiguous.
 *   k_new/v_new  [B, Lnew, Hkv, D] contiguous, or NULL with Lnew == 0.
 *   cache_seqlens int32 [B] (device): tokens already cached.
 *   block_table  int32 [B, >= max_pages] (row stride bt_stride) or NULL for a
 *                contiguous cache; entries past ceil(Lk_b/page_size) are never
 *                read.  page_size: see pa_tensor4.
 *   cache_extent paged: pages in the pool; contiguous: tokens per sequence.
 *   max_seqlen_k host-known upper bound of Lk_b (a capacity, never read back).
 *   scale        softmax scale (e.g. 1/sqrt(D)).
 *   num_splits   0: split-KV count chosen on the GPU from cache_seqlens;
 *                >= 1: at most that many splits per sequence.
 *   out          [B, Lq, Hq, D] contiguous; lse fp32 [B, Hq, Lq] or NULL.
 *   workspace    device scratch of pa_fwd_kvcache_workspace_size(...) bytes
 *                (may be NULL when that size is 0).  Its contents on entry do
 *                not matter.
 * Which kernel runs depends on the query rows per kv head, Lq * (Hq / Hkv):
 *   <= 2     the split-KV decode kernel, CUDA-core consumers;
 *   3 - 16   the split-KV decode kernel, warp-level tensor-core consumer;
 *   17 - 128 the tcgen05 engine, all query heads of a kv head packed in one
 *            tile, split-KV, followed by the combine kernel when it splits;
 *   > 128    the tcgen05 prefill kernel, two 128-row query tiles per CTA.
 * The decode kernel appends k_new / v_new in the same launch and merges its
 * splits in the same launch (one launch per call); the engine and prefill
 * paths run the append kernel first.
 */
PA_API int pa_fwd_kvcache(const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                          pa_tensor4 k_cache, pa_tensor4 v_cache, const void* k_new,
                          const void* v_new, int Lnew, const int32_t* cache_seqlens,
                          const int32_t* block_table, int64_t bt_stride, int max_pages,
                          int page_size, int B, int Lq, int Hq, int Hkv, int D,
                          int64_t cache_extent, int max_seqlen_k,
                          float scale, int causal, int num_splits, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, int32_t* err_word, int dtype,
                          pa_stream_t stream);

/* Bytes of workspace pa_fwd_kvcache needs for these sizes (0 if none). */
PA_API size_t pa_fwd_kvcache_workspace_size(int B, int Lq, int Hq, int Hkv, int D,
                                            int max_seqlen_k, int num_splits);

/*
 * pa_fwd_kvcache_rotary -- pa_fwd_kvcache with rotary position embedding of
 * the new tokens.  flash-attention #824 "Add support for small page sizes"
 * names the feature (a fix to fused RoPE embeddings in this forward) without
 * defining it; the rotation is the published RoFormer one:
 *
 *   - features [0, rotary_dim) are rotated, the rest pass through;
 *   - rotary_interleaved == 0: feature p pairs with p + rotary_dim / 2;
 *     otherwise feature 2p pairs with 2p + 1;
 *   - a pair (x1, x2) of a token at position pos becomes
 *     (x1 c - x2 s, x1 s + x2 c), c = rotary_cos[pos][p], s = rotary_sin[pos][p].
 *
 * Positions: new token i of sequence b is at cache_seqlens[b] + i (the slot the
 * append writes it to); query row i of Lq is at cache_seqlens[b] + Lnew - Lq + i.
 * The rotated k is what the append stores in the cache; the rotated q is what
 * attends.  The rotation is computed in fp32 and rounded once to the dtype.
 *
 * Arguments are those of pa_fwd_kvcache plus
 *   rotary_cos, rotary_sin  [rotary_len, rotary_dim / 2], row-major, dtype of q;
 *                           device memory owned by the caller.
 *   rotary_len              rows of the tables; a position >= rotary_len
 *                           leaves the token unrotated and records
 *                           PA_DEVERR_LENGTH (sequence, position) in err_word.
 *   rotary_dim              even, 2 <= rotary_dim <= D.
 * Requires Lnew >= 1 (the rotation applies to appended tokens).  workspace:
 * pa_fwd_kvcache_rotary_workspace_size bytes, 256-byte aligned.
 * Query blocks of up to 16 rows per kv head (Lq * Hq / Hkv <= 16: decode,
 * GQA decode, short multi-query decode) are rotated inside the attention
 * launch: q as it is staged for the kernel, k_new where the fused append
 * stores it; the workspace is then pa_fwd_kvcache's own.  Longer query
 * blocks run one extra kernel (the rotation into the workspace, ahead of
 * pa_fwd_kvcache's own scratch) before the attention launches.  Same return
 * codes as pa_fwd_kvcache.
 */
PA_API int pa_fwd_kvcache_rotary(const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                                 pa_tensor4 k_cache, pa_tensor4 v_cache, const void* k_new,
                                 const void* v_new, int Lnew, const int32_t* cache_seqlens,
                                 const int32_t* block_table, int64_t bt_stride, int max_pages,
                                 int page_size, int B, int Lq, int Hq, int Hkv, int D,
                                 int64_t cache_extent, int max_seqlen_k, const void* rotary_cos,
                                 const void* rotary_sin,
                                 int rotary_len, int rotary_dim, int rotary_interleaved,
                                 float scale, int causal, int num_splits, void* out, float* lse,
                                 void* workspace, size_t workspace_bytes, int32_t* err_word,
                                 int dtype, pa_stream_t stream);

/* Bytes of workspace pa_fwd_kvcache_rotary needs for these sizes. */
PA_API size_t pa_fwd_kvcache_rotary_workspace_size(int B, int Lq, int Hq, int Hkv, int D, int Lnew,
                                                   int max_seqlen_k, int num_splits);

/*
 * pa_fwd_kvcache_noalloc -- pa_fwd_kvcache for callers that cannot allocate
 * device memory.  (No counterpart on the pages: this is a library-usage entry
 * point, not part of the attention method.)
 *
 * Some callers cannot call cudaMalloc: code running inside another library's
 * allocator or stream callback, serving processes whose device memory pool is
 * owned and capped by the framework, or latency paths that must never reach
 * the driver's allocator.  They can pass inputs and outputs but not the
 * split-KV scratch that pa_fwd_kvcache takes as `workspace`.  This variant
 * takes the same arguments minus the workspace and uses a fixed scratch array
 * of PA_NOALLOC_SCRATCH_BYTES that every GPU using the library holds until the
 * process exits.  It calls no allocating routine.
 *
 *   - Sizes whose split scratch (pa_fwd_kvcache_workspace_size) exceeds
 *     PA_NOALLOC_SCRATCH_BYTES are rejected with PA_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current).  Under CUDA's lazy module
 *     loading that lookup may load the library's device code on that device,
 *     which allocates in the driver (the array included): make the first call
 *     during set-up -- outside allocator hooks and before any stream capture.
 *   - All calls share the array, which keeps the last call's contents; no
 *     entry needs to start at zero.  Calls whose kernels overlap on the GPU
 *     (other streams, other threads) race on it: serialise them.
 */
#define PA_NOALLOC_SCRATCH_BYTES (8 << 20)
PA_API int pa_fwd_kvcache_noalloc(const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                                  pa_tensor4 k_cache, pa_tensor4 v_cache, const void* k_new,
                                  const void* v_new, int Lnew, const int32_t* cache_seqlens,
                                  const int32_t* block_table, int64_t bt_stride, int max_pages,
                                  int page_size,
                                  int B, int Lq, int Hq, int Hkv, int D, int64_t cache_extent,
                                  int max_seqlen_k, float scale, int causal, int num_splits,
                                  void* out, float* lse, int32_t* err_word, int dtype,
                                  pa_stream_t stream);

/*
 * pa_fwd_varlen_unified -- one launch for a mixed batch of chunked-prefill
 * and decode sequences over a paged cache (vLLM #6052 "Unify the kernel used
 * in flash attention backend": a single varlen kernel for prefill, decode and
 * chunked prefill; cumulative query lengths padded with repeated entries).
 *
 *   q             [total_q, Hq, D], element strides q_st, q_sh; packed by
 *                 cu_seqlens_q.
 *   cu_seqlens_q  int32 [B+1], non-decreasing, cu_seqlens_q[0] == 0.  A
 *                 sequence with no query rows (a padding entry) writes nothing.
 *   seqlens_k     int32 [B]: keys of sequence b, INCLUDING its new chunk,
 *                 which must already be in the cache (pa_append_kv).
 *   max_seqlen_q, max_seqlen_k  host-known capacities (grid sizing only).
 *   out [total_q, Hq, D] contiguous; lse fp32 [Hq, total_q] or NULL.
 *   workspace     pa_fwd_varlen_workspace_size(...) bytes.
 * The tcgen05 engine runs the whole batch in one launch: sequences of up to
 * 128 query rows per kv head as packed (split-KV) items, longer chunks as
 * pairs of 128-row query tiles, each CTA taking a contiguous run of work
 * units of equal estimated cost; when a decode sequence is split, the combine
 * kernel follows as a programmatic dependent launch.  At most 4096 entries
 * (B, padding entries included); more return PA_ERR_UNSUPPORTED.
 */
PA_API int pa_fwd_varlen_unified(const void* q, int64_t q_st, int64_t q_sh, pa_tensor4 k_cache,
                                 pa_tensor4 v_cache, const int32_t* cu_seqlens_q,
                                 const int32_t* seqlens_k, const int32_t* block_table,
                                 int64_t bt_stride, int max_pages, int page_size, int B,
                                 int total_q,
                                 int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                                 int64_t num_pages, float scale, int causal, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 int32_t* err_word, int dtype, pa_stream_t stream);

PA_API size_t pa_fwd_varlen_workspace_size(int B, int total_q, int max_seqlen_q, int Hq,
                                           int Hkv, int D, int max_seqlen_k);

/*
 * pa_split_combine -- merge split-KV partial results (the combine step that
 * follows flash_fwd_splitkv_kernel, vLLM #6052 comment on num_splits == 0 with
 * a page table; flash-attention #1000).
 *
 * For each b < B, query row i < Lq, head h < Hq with n = splits_per_seq[b]
 * (or S when splits_per_seq == NULL):
 *   LSE = ln sum_{s<n} exp(LSE_s),  O = sum_{s<n} exp(LSE_s - LSE) O_s,
 * where O_s = o_partial[s, b, i, h, :] is the NORMALISED output of split s
 * and LSE_s = lse_partial[s, b, i, h] (-inf for an empty split, whose O_s is
 * then never read).  Rows whose n is 0 are left untouched; n is clamped to S.
 *   o_partial fp32 [S, B, Lq, Hq, D]; lse_partial fp32 [S, B, Lq, Hq];
 *   out [B, Lq, Hq, D] (dtype); lse fp32 [B, Hq, Lq] or NULL.
 */
PA_API int pa_split_combine(const float* o_partial, const float* lse_partial,
                            const int32_t* splits_per_seq, int S, int B, int Lq, int Hq, int D,
                            void* out, float* lse, int dtype, pa_stream_t stream);

/* Human-readable text of the last non-OK return on the calling thread. */
PA_API const char* pa_last_error_string(void);

/* Library version, major * 10000 + minor * 100 + patch. */
PA_API int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
