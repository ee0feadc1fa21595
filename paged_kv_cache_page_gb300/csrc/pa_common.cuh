// Device-side building blocks shared by the paged-attention kernels (sm_103a):
// mbarrier pipeline primitives with bounded waits, TMA tensor loads, fast
// exp2/log2, element-type traits, error reporting and the device split-KV
// schedule.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedattn.h"
#include "pa_internal.h"

namespace pa {
// A pipeline wait that has not completed after this long is treated as a
// failure: the kernel records PA_DEVERR_TIMEOUT and finishes without waiting.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------- element types
template <typename T> struct Elem;
template <> struct Elem<__half> {
  using T2 = __half2;
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
  }
  static __device__ __forceinline__ uint32_t from_f2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ __half from_f(float a) { return __float2half_rn(a); }
};
template <> struct Elem<__nv_bfloat16> {
  using T2 = __nv_bfloat162;
  static __device__ __forceinline__ float2 to_f2(uint32_t u) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(h);
  }
  static __device__ __forceinline__ uint32_t from_f2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  static __device__ __forceinline__ __nv_bfloat16 from_f(float a) { return __float2bfloat16_rn(a); }
};

// ---------------------------------------------------------------- math
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float neg_inf() { return __int_as_float(0xff800000); }

// ---------------------------------------------------------------- errors
__device__ __forceinline__ void report(int32_t* err, int code, int b, int value) {
  if (err == nullptr) return;
  if (atomicCAS(err, 0, code) == 0) {
    err[1] = b;
    err[2] = value;
  }
}

// ---------------------------------------------------------------- timers
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Announces `bytes` more transaction bytes for the current phase without
// arriving (the caller arrives separately).
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Both tests in one block, so that the second is issued before the first
// returns: one round trip instead of two when both phases are complete.
__device__ __forceinline__ bool mbar_try_wait2(uint64_t* bar0, uint32_t parity0, uint64_t* bar1,
                                               uint32_t parity1) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 q, [%3], %4;\n\t"
      "and.pred p, p, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar0)), "r"(parity0), "r"(smem_u32(bar1)), "r"(parity1)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of parity `parity` to complete.  Returns false
// (and never blocks longer than kWaitTimeoutNs) if it does not.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > kWaitTimeoutNs) return false;
  }
  return true;
}

// Programmatic dependent launch: a grid lets the next (dependent) grid of its
// stream be scheduled once all its CTAs have executed launch_dependents; the
// dependent grid's griddep_wait returns when this grid has completed and its
// memory writes are visible.  Both are no-ops without such a launch.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA / tensor core) accesses of the same locations.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier over `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 4-D tiled bulk tensor load global -> shared, completion signalled on `bar`
// as transaction bytes.  c0 is the innermost (head_dim) coordinate and is
// always 0 or a multiple of 64 elements here, which keeps it 16-byte aligned.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
// Untiled bulk copy global -> shared, completing `bytes` on `bar`: both
// addresses 16-byte aligned, `bytes` a multiple of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- page resolution
// Where the 16-token box `lp` (tokens [16 lp, 16 lp + 16)) of sequence `b`
// lives, as TMA coordinates (row coordinate c2, page-or-sequence coordinate
// c3) and as an element offset of its first token slot for head 0.  Pages of
// P = 16 << page_shift tokens hold 1 << page_shift boxes: the box is in the
// page of table entry lp >> page_shift, at row 16 (lp mod (1 << page_shift)).
// The page is resolved absolutely for every iteration (never by a delta from
// the previous page), and the table is never indexed at or beyond
// `max_pages`.
struct PageRef {
  int c2, c3;
  int64_t elem_off;  // offset of slot 0, head 0 (element units) in the K cache view
  bool ok;           // false: entry out of range (reads use page 0, writes skipped)
};

struct CacheGeom {
  const int32_t* block_table;  // nullptr: contiguous cache
  int64_t bt_stride;
  int max_pages;      // table width (paged)
  int64_t extent;     // pages in pool (paged) or tokens per sequence (contiguous)
  int64_t sb, st;     // element strides of the K cache (V uses its own strides)
  int page_shift;     // log2(page size / 16) (paged)
};

__device__ __forceinline__ PageRef resolve_page(const CacheGeom& g, int b, int lp) {
  PageRef r;
  if (g.block_table != nullptr) {
    int phys = 0;
    const int entry = lp >> g.page_shift;
    bool ok = lp >= 0 && entry < g.max_pages;
    if (ok) phys = __ldg(g.block_table + (int64_t)b * g.bt_stride + entry);
    ok = ok && phys >= 0 && (int64_t)phys < g.extent;
    if (!ok) phys = 0;
    r.c2 = ok ? (lp & ((1 << g.page_shift) - 1)) * kPage : 0;
    r.c3 = phys;
    r.elem_off = (int64_t)phys * g.sb + (int64_t)r.c2 * g.st;
    r.ok = ok;
  } else {
    // Rows past the capacity in the last box are zero-filled by the TMA unit
    // and never written; only the box start must lie inside the cache.
    const int64_t row = (int64_t)lp * kPage;
    const bool ok = lp >= 0 && row < g.extent;
    r.c2 = ok ? (int)row : 0;
    r.c3 = b;
    r.elem_off = (int64_t)b * g.sb + (ok ? row : 0) * g.st;
    r.ok = ok;
  }
  return r;
}

// ---------------------------------------------------------------- split-KV schedule
// Pages per split when a sequence of `pages` pages is cut into splits of at
// most `chunk` pages (rounded up to 4 pages, at most s_max splits); writes
// the split count.  With s_max <= 1 (or no pages) there is one split.
struct SplitSched {
  int s_max;
  int target_ctas;      // kForcedSplitTarget: explicit split count (uniform splits)
  int min_chunk_pages;  // smallest split (automatic splits)
};

constexpr int kForcedSplitTarget = 1 << 30;

__device__ __forceinline__ int round_up4(int x) { return (x + 3) & ~3; }

__device__ __forceinline__ int split_pages_per(const SplitSched& s, int pages, int chunk,
                                               int* n_out) {
  if (s.s_max <= 1 || pages <= 0) {
    *n_out = 1;
    return pages > 0 ? pages : 0;
  }
  int n = (pages + chunk - 1) / chunk;
  if (n < 1) n = 1;
  if (n > s.s_max) n = s.s_max;
  int per = round_up4((pages + n - 1) / n);
  n = (pages + per - 1) / per;
  *n_out = n;
  return per;
}

}  // namespace pa
