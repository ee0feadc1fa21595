// Internal declarations of the persistent tensor-core attention engine
// (prefill tiles, packed GQA/decode items and mixed varlen batches).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kEngineMaxB = 4096;  // sequences a launch with a per-sequence schedule may hold
constexpr int kEngineMaxRows = 128;

struct EngineParams {
  void* out;    // [rows, Hq, D] with rows = B*Lq (kvcache) or total_q (varlen)
  float* lse;   // kvcache: [B, Hq, Lq]; varlen: [Hq, total_q]; may be null
  const int32_t* cache_seqlens;  // kvcache: keys already cached (Lk = that + Lnew)
  int Lnew;
  const int32_t* cu_seqlens_q;   // varlen (non-null selects it)
  const int32_t* seqlens_k;
  const int32_t* block_table;    // null: contiguous cache
  int64_t bt_stride;
  int max_pages;
  int page_shift;                // log2(page size / 16): 16-token boxes per table entry
  int64_t extent;                // pages in pool, or tokens per sequence
  int B, Lq, Hq, Hkv, G, max_seqlen_k, total_q;
  int pack_rows;   // sequences with q_len * G <= pack_rows run as packed items (one per kv head
                   // and split); longer ones as 128-row query tiles of one head
  int max_q_tiles; // host-known bound of query tiles per sequence (uniform kvcache mode)
  float scale_log2;
  int causal;
  int s_max, target_ctas, min_chunk_pages;  // split plan of packed items
  int tilebal;       // kvcache packed call with automatic splits: every CTA takes an equal share
                     // of the concatenated (sequence, kv head) streams' key tiles, cutting
                     // streams at the share boundaries; split counts are kept per stream
  float* o_part;     // [s_max, rows, Hq, D] normalised split outputs
  float* lse_part;   // [s_max, rows, Hq]
  int32_t* nsplit;   // [B], or [B, Hkv] under tilebal: splits to combine (0: final output
                     // written directly)
  int32_t* err;
};

// tm_q1: q map with box {64, 1, 128, 1} (one head, 128 rows); tm_q2: box
// {64, G, 128/G, 1} (the G heads of one kv head, packed rows); tm_k/tm_v:
// cache maps with box {64, 1, 16, 1}; all 128-byte swizzled.  `grid` CTAs.
cudaError_t launch_engine(const EngineParams& p, const CUtensorMap& tm_q1,
                          const CUtensorMap& tm_q2, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, int D, int dtype, int grid, cudaStream_t st);
int engine_grid();

// Prefill of a kvcache call whose query blocks are longer than one packed tile
// (uniform query length Lq, cu_seqlens_q == null): two 128-row query tiles of
// one head per CTA sharing every K/V tile.  Uses p.out, p.lse, the sequence
// and cache fields, scale_log2 and causal; the split fields are ignored.
// tm_q: q map with box {64, 1, 128, 1}; tm_k/tm_v as for launch_engine.
cudaError_t launch_prefill(const EngineParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, int D, int dtype, cudaStream_t st);

}  // namespace pa
