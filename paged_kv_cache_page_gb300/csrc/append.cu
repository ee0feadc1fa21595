// Standalone KV append (sm_103a): bit copy of new tokens' k/v into their cache
// slots through the block table -- the k=/v= write of flash_attn_with_kvcache
// (flash-attention #824 "Add support for small page sizes": the call writes
// through block_table and allocates nothing) and the separate cache-write op
// that vLLM #3010 "Introduce flash-attn" benchmarks next to the fused one.
// One thread per 16-byte chunk of a (token, head) row: fully coalesced reads
// of k_new/v_new and 16-byte writes into the (strided) cache rows.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  const int chunks = p.D / 8;  // 16-byte chunks per row
  const long long total = (long long)p.B * p.Lnew * p.Hkv * chunks;
  CacheGeom geom{p.block_table, p.bt_stride, p.max_pages, p.extent, p.k_sb, p.k_st, p.page_shift};
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int c = (int)(idx % chunks);
    long long r = idx / chunks;
    const int g = (int)(r % p.Hkv);
    r /= p.Hkv;
    const int i = (int)(r % p.Lnew);
    const int b = (int)(r / p.Lnew);
    const int old = __ldg(p.cache_seqlens + b);
    const long long pos = (long long)old + i;
    const bool len_ok = old >= 0 &&
                        (p.block_table != nullptr ? ((pos / kPage) >> p.page_shift) < p.max_pages
                                                  : pos < p.extent);
    if (!len_ok) {
      if (g == 0 && c == 0) report(p.err, PA_DEVERR_LENGTH, b, (int)pos);
      continue;
    }
    const PageRef ref = resolve_page(geom, b, (int)(pos / kPage));
    if (!ref.ok) {
      if (g == 0 && c == 0) report(p.err, PA_DEVERR_PAGE_OOB, b, (int)(pos / kPage));
      continue;
    }
    const int slot = (int)(pos % kPage);
    const long long src = (((long long)b * p.Lnew + i) * p.Hkv + g) * p.D + c * 8;
    const uint4 kv = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.k_new) + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.v_new) + src));
    uint16_t* kd = reinterpret_cast<uint16_t*>(p.k_cache) + (long long)ref.c3 * p.k_sb +
                   (long long)(ref.c2 + slot) * p.k_st + (long long)g * p.k_sh + c * 8;
    uint16_t* vd = reinterpret_cast<uint16_t*>(p.v_cache) + (long long)ref.c3 * p.v_sb +
                   (long long)(ref.c2 + slot) * p.v_st + (long long)g * p.v_sh + c * 8;
    *reinterpret_cast<uint4*>(kd) = kv;
    *reinterpret_cast<uint4*>(vd) = vv;
  }
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, cudaStream_t st) {
  const long long total = (long long)p.B * p.Lnew * p.Hkv * (p.D / 8);
  if (total <= 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  const long long cap = 152LL * 8;
  if (blocks > cap) blocks = cap;
  append_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
