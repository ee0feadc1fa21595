// pa_fwd_kvcache_noalloc: the kvcache forward for callers that cannot
// allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is off limits -- inside a
// host callback or another library's allocator hook, in a process whose
// memory pool is owned and capped by a serving framework, or in a tight
// latency path that must never hit the driver's allocator.  Such a caller can
// pass its own inputs and outputs but cannot provide the split-KV scratch that
// pa_fwd_kvcache takes as `workspace`.
//
// Here that scratch is a fixed array in device memory: every GPU on which the
// library's device code is loaded holds PA_NOALLOC_SCRATCH_BYTES of it until
// the process exits.  The entry point itself calls no cudaMalloc, cudaFree or
// allocating library routine.
//
// Host code cannot use the array's name as a device pointer (on the host it
// names a shadow object), so the device address is looked up once per device
// with cudaGetSymbolAddress, with that device current, on the first call made
// on it.  With CUDA's lazy module loading (the default) that lookup may be
// what loads the library's device code on the device, and loading allocates
// in the driver, the array included.  The first call on each device should
// therefore be made during set-up: outside any allocator hook and before any
// stream capture.
//
// All calls share the one array and it keeps the last call's contents.
// Nothing in it has to start at zero (each call writes every scratch entry it
// later reads), but two calls whose kernels overlap on the GPU -- on different
// streams, or from different threads -- race on it and must be serialised by
// the caller.
#include <mutex>

#include "pa_internal.h"

namespace pa {
// Records a message for pa_last_error_string() (defined in api.cu).
int set_error(int code, const char* fmt, ...);
}  // namespace pa

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up on the
// first call per device).  Returns nullptr and fills `err` on failure.
void* scratch_on_current_device(cudaError_t* err) {
  int dev = -1;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (*err != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  *err = cudaSuccess;
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

PA_API int pa_fwd_kvcache_noalloc(const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                                  pa_tensor4 k_cache, pa_tensor4 v_cache, const void* k_new,
                                  const void* v_new, int Lnew, const int32_t* cache_seqlens,
                                  const int32_t* block_table, int64_t bt_stride, int max_pages,
                                  int page_size, int B, int Lq, int Hq, int Hkv, int D,
                                  int64_t cache_extent,
                                  int max_seqlen_k, float scale, int causal, int num_splits,
                                  void* out, float* lse, int32_t* err_word, int dtype,
                                  pa_stream_t stream) {
  const size_t need =
      pa_fwd_kvcache_workspace_size(B, Lq, Hq, Hkv, D, max_seqlen_k, num_splits);
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES)
    return pa::set_error(PA_ERR_WORKSPACE,
                         "pa_fwd_kvcache_noalloc: these sizes need %zu bytes of split scratch, "
                         "more than its fixed %d bytes; lower num_splits or use pa_fwd_kvcache "
                         "with a caller-provided workspace",
                         need, (int)PA_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (need > 0) {
    cudaError_t e = cudaSuccess;
    scratch = scratch_on_current_device(&e);
    if (scratch == nullptr)
      return pa::set_error(PA_ERR_CUDA, "pa_fwd_kvcache_noalloc: scratch address lookup: %s",
                           cudaGetErrorString(e));
  }
  return pa_fwd_kvcache(q, q_sb, q_st, q_sh, k_cache, v_cache, k_new, v_new, Lnew,
                        cache_seqlens, block_table, bt_stride, max_pages, page_size, B, Lq, Hq,
                        Hkv, D,
                        cache_extent, max_seqlen_k, scale, causal, num_splits, out, lse, scratch,
                        need, err_word, dtype, stream);
}

}  // extern "C"
