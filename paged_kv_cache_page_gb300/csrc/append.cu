// Standalone KV append (sm_103a): bit copy of new tokens' k/v into their cache
// slots through the block table -- the k=/v= write of flash_attn_with_kvcache
// (flash-attention #824 "Add support for small page sizes": the call writes
// through block_table and allocates nothing) and the separate cache-write op
// that vLLM #3010 "Introduce flash-attn" benchmarks next to the fused one.
// A block takes (sequence, token) rows in turn: the row's slot is resolved
// once (a block-table read) and its threads copy the row's Hkv x D/8 16-byte
// chunks of k and of v -- coalesced reads of k_new/v_new, 16-byte writes into
// the (strided) cache rows -- with no per-chunk index division.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  const int chunk_shift = p.D == 128 ? 4 : 3;  // log2(16-byte chunks per head row)
  const int row_chunks = p.Hkv << chunk_shift;
  const long long rows = (long long)p.B * p.Lnew;
  CacheGeom geom{p.block_table, p.bt_stride, p.max_pages, p.extent, p.k_sb, p.k_st, p.page_shift};
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const int i = (int)(r % p.Lnew);
    const int b = (int)(r / p.Lnew);
    const int old = __ldg(p.cache_seqlens + b);
    const long long pos = (long long)old + i;
    const bool len_ok = old >= 0 &&
                        (p.block_table != nullptr ? ((pos / kPage) >> p.page_shift) < p.max_pages
                                                  : pos < p.extent);
    if (!len_ok) {
      if (threadIdx.x == 0) report(p.err, PA_DEVERR_LENGTH, b, (int)pos);
      continue;
    }
    const PageRef ref = resolve_page(geom, b, (int)(pos / kPage));
    if (!ref.ok) {
      if (threadIdx.x == 0) report(p.err, PA_DEVERR_PAGE_OOB, b, (int)(pos / kPage));
      continue;
    }
    const long long row = ref.c2 + pos % kPage;  // slot within the page (or the sequence row)
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(p.k_new) + r * ((long long)p.Hkv * p.D);
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(p.v_new) + r * ((long long)p.Hkv * p.D);
    uint16_t* kd = reinterpret_cast<uint16_t*>(p.k_cache) + (long long)ref.c3 * p.k_sb + row * p.k_st;
    uint16_t* vd = reinterpret_cast<uint16_t*>(p.v_cache) + (long long)ref.c3 * p.v_sb + row * p.v_st;
    for (int e = threadIdx.x; e < row_chunks; e += blockDim.x) {
      const int g = e >> chunk_shift;
      const int c = (e & ((1 << chunk_shift) - 1)) * 8;
      const uint4 kv = __ldg(reinterpret_cast<const uint4*>(ks + g * p.D + c));
      const uint4 vv = __ldg(reinterpret_cast<const uint4*>(vs + g * p.D + c));
      *reinterpret_cast<uint4*>(kd + (long long)g * p.k_sh + c) = kv;
      *reinterpret_cast<uint4*>(vd + (long long)g * p.v_sh + c) = vv;
    }
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t st) {
  const long long rows = (long long)p.B * p.Lnew;
  if (rows <= 0 || p.Hkv <= 0) return cudaSuccess;
  long long blocks = rows;
  const long long cap = 152LL * 8;  // 8 resident blocks of 256 threads per SM
  if (blocks > cap) blocks = cap;
  append_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
