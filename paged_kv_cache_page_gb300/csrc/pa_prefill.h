// Internal declarations of the tensor-core prefill path.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// One CTA = one 128-row query tile of one query head of one sequence.
struct PrefillParams {
  void* out;    // kvcache: [B, Lq, Hq, D]; varlen: [total_q, Hq, D]
  float* lse;   // kvcache: [B, Hq, Lq]; varlen: [Hq, total_q]; may be null
  const int32_t* cache_seqlens;  // kvcache: keys already cached (Lk = that + Lnew)
  int Lnew;
  const int32_t* cu_seqlens_q;   // varlen (non-null selects it)
  const int32_t* seqlens_k;
  const int32_t* block_table;    // null: contiguous cache
  int64_t bt_stride;
  int max_pages;
  int64_t extent;                // pages in pool, or tokens per sequence
  int B, Lq, Hq, Hkv, G, max_seqlen_k, total_q;
  int q_tiles;                   // query tiles per sequence (from the host-known max)
  int decode_rows;               // varlen: sequences with q_len * G <= this are left to the decode path
  float scale_log2;
  int causal;
  int32_t* err;
};

// tm_q: 4-D map of q with box {64, 1, 128, 1}; tm_k/tm_v: cache maps with box
// {64, 1, 16, 1}; all with 128-byte swizzle.
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tm_q,
                           const CUtensorMap& tm_k, const CUtensorMap& tm_v, int D, int dtype,
                           cudaStream_t st);

}  // namespace pa
