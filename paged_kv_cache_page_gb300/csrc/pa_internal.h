// Internal (non-exported) declarations shared by the host-side API and the
// kernel translation units of libpagedattn.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedattn.h"

namespace pa {

constexpr int kPage = 16;  // tokens per page
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Parameters of the split-KV decode path.  Rows of one work item are the
// Lq * G query rows that share one kv head of one sequence.
struct DecodeParams {
  const void* q;
  int64_t q_sb, q_st, q_sh;  // element strides of [B, Lq, Hq, D]
  void* out;                 // [B, Lq, Hq, D]
  float* lse;                // [B, Hq, Lq]; may be null
  const void* k_new;         // [B, Lnew, Hkv, D] or null
  const void* v_new;
  int Lnew;
  void* k_cache;
  void* v_cache;
  int64_t k_sb, k_st, k_sh, v_sb, v_st, v_sh;
  const int32_t* block_table;  // null: contiguous cache
  int64_t bt_stride;
  int max_pages;
  int page_shift;  // log2(page size / 16): 16-token boxes per table entry = 1 << page_shift
  int64_t extent;  // pages in pool, or tokens per sequence (contiguous)
  const int32_t* cache_seqlens;  // [B] keys already cached
  int B, Lq, Hq, Hkv, G, max_seqlen_k;
  float scale_log2;  // softmax scale * log2(e)
  int causal;
  int s_max, target_ctas, min_chunk_pages;
  int grid_ctas;     // persistent CTAs launched (resident capacity)
  float* o_part;     // [s_max, B * Lq, Hq, D]
  float* lse_part;   // [s_max, B * Lq, Hq]
  // [B, Hkv] arrival words of the in-launch split merge: (launch tag, count)
  unsigned long long* split_ctr;
  int32_t* err;
  // rotary embedding of the new tokens (rot_cos == null: none): features
  // [0, rot_dim) of q and of k_new rotated at their positions, pairs
  // (p, p + rot_dim / 2) or, interleaved, (2p, 2p + 1); tables
  // [rot_len, rot_dim / 2] of the q dtype
  const void* rot_cos;
  const void* rot_sin;
  int rot_dim, rot_len, rot_interleaved;
};

struct CombineParams {
  const float* o_part;
  const float* lse_part;
  const int32_t* nsplit;  // null: all S splits valid; else entry
                          // b * ns_stride + h / ns_group is the split count of (b, h)
  int ns_stride, ns_group;
  int S, B, Lq, Hq;
  const int32_t* cu_seqlens_q;  // non-null: varlen row addressing
  int total_q;
  void* out;
  float* lse;
};

struct AppendParams {
  void* k_cache;
  void* v_cache;
  int64_t k_sb, k_st, k_sh, v_sb, v_st, v_sh;
  const void* k_new;
  const void* v_new;
  const int32_t* cache_seqlens;
  const int32_t* block_table;
  int64_t bt_stride;
  int max_pages;
  int page_shift;  // log2(page size / 16)
  int64_t extent;
  int B, Lnew, Hkv, D;
  int32_t* err;
};

// Launchers (each defined in the .cu file that holds its kernel).  They
// return a cudaError_t from the launch.
cudaError_t launch_append(const AppendParams& p, cudaStream_t st);

// Rotary embedding of a kvcache call's new tokens into scratch copies of q
// (contiguous [B, Lq, Hq, D]) and k_new ([B, Lnew, Hkv, D]).
struct RotaryParams {
  const void* q;
  int64_t q_sb, q_st, q_sh;
  const void* k_new;
  void* q_out;
  void* k_out;
  const void* cos;  // [rotary_len, rotary_dim / 2], the q / cache dtype
  const void* sin;
  const int32_t* cache_seqlens;
  int B, Lq, Lnew, Hq, Hkv, D, rotary_dim, rotary_len, interleaved;
  int32_t* err;
};
cudaError_t launch_rotary(const RotaryParams& p, int dtype, cudaStream_t st);
// `dependent`: launched as a programmatic dependent of the kernel just
// enqueued on `st` (its blocks may be scheduled while that kernel drains and
// wait on the device until it has completed and its writes are visible).
cudaError_t launch_combine(const CombineParams& p, int D, int dtype, int rows_total,
                           cudaStream_t st, bool dependent = false);
// Decode: `rmax` in {1, 2, 8, 16} (rows per kv head, rounded up).  tmk/tmv
// are 4-D tensor maps of the caches with box {D, 1, 16, 1} unswizzled (rmax
// 1, 2) or {64, 1, 16, 1} with the 128-byte swizzle (rmax 8, 16).
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          int D, int dtype, int rmax, cudaStream_t st);
// Resident CTAs per SM of the decode kernel for this configuration (0 on error).
int decode_ctas_per_sm(int D, int dtype, int rmax);
constexpr int kDecodeMaxRows = 16;
constexpr int kDecodeMaxSchedB = 512;

// Host helpers (api.cu).
int num_sms();
bool encode_cache_map(CUtensorMap* map, const void* base, int dtype, int D, int Hkv, int64_t dim2,
                      int64_t dim3, int64_t stride_h, int64_t stride_t, int64_t stride_b,
                      int box_d, int box_rows, bool swizzle128);

}  // namespace pa
