// C ABI of libpagedattn.so: argument validation, tensor-map encoding, the
// host half of the split-KV plan (capacities only -- lengths stay on the GPU),
// and kernel launches.  No function here synchronises or allocates.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "pa_internal.h"
#include "pa_engine.h"

namespace pa {
namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tokens per page of a paged cache: 16 << shift with shift in [0, 4] (16 to 256
// tokens, the 16-token pages of vLLM and the 256-token ones flash-attention
// required, vLLM #3010).  The kernels move 16-token boxes; a page holds
// 1 << shift of them.  Returns false for other sizes.
bool page_shift_of(int page_size, int* shift) {
  for (int s = 0; s <= 4; ++s)
    if (page_size == (kPage << s)) {
      *shift = s;
      return true;
    }
  return false;
}
bool mult8(int64_t s) { return s > 0 && (s % 8) == 0; }

// Split-KV planning constants.  The host only fixes a cap on splits per
// sequence from capacities; the GPU picks the actual counts from the lengths.
constexpr int kSplitCapTargetCtas = 304;  // 152 SMs x 2 resident decode CTAs
constexpr int kMinChunkPages = 8;         // each split streams >= 128 keys
constexpr int kMaxSplits = 128;
// Query blocks of at most this many rows per kv head run on the split-KV
// decode kernel (1-2 rows: CUDA-core consumers; 3-16: warp-level tensor-core
// consumer); larger ones on the tcgen05 engine.
constexpr int kCudaCoreRows = 16;

int plan_s_max(int B, int Hkv, int max_seqlen_k, int num_splits) {
  const int max_pages = std::max(1, (max_seqlen_k + kPage - 1) / kPage);
  // The device schedule keeps one prefix entry per sequence in shared memory;
  // batches beyond that table run unsplit (they have parallelism to spare).
  if (num_splits == 1 || B > kDecodeMaxSchedB) return 1;
  if (num_splits > 1) return std::min(std::min(num_splits, kMaxSplits), max_pages);
  if ((long long)B * Hkv >= 4LL * kSplitCapTargetCtas) return 1;
  int s = (max_pages + kMinChunkPages - 1) / kMinChunkPages;
  s = std::min(s, kSplitCapTargetCtas / std::max(1, Hkv) + 1);
  s = std::min(s, kMaxSplits);
  return std::max(1, s);
}

// Host gate of the automatic split: may the device's balanced schedule (equal
// page shares over all streams, see decode.cu) pay for its partial writes
// and in-launch merge, for B sequences of the capacity max_seqlen_k?  When it
// cannot, the call runs one split per stream (no schedule, no partials).
// Two tests, both on capacities only:
//   - whole splits per sequence: the cheapest of n in {1..16} splits per
//     stream, costed as rounds of items over the resident CTAs times (pages
//     per item + 4); a split plan must beat the unsplit one by 3 % (its
//     one-unit wins, such as a 32-page capacity cut in four, do not pay);
//   - balance: streams of at least 128 pages (2048 keys) whose unsplit last
//     round leaves at least a tenth of the CTA rounds idle, when equal shares
//     save at least 32 pages per CTA (measured, 32 kv heads: ctx 4096 x B8
//     and ctx 2048 x B16 save 40 pages and run 3.6 / 4.2 % faster; ctx 2048
//     x B8 saves 20 and runs 7 % slower, the split's fixed cost).
bool decode_splits_useful(int B, int Hkv, int max_seqlen_k, int s_max, int target_ctas) {
  if (s_max <= 1 || target_ctas < 1) return false;
  const int P = std::max(1, (max_seqlen_k + kPage - 1) / kPage);
  const int cands[8] = {1, 2, 3, 4, 6, 8, 12, 16};
  auto up4 = [](int x) { return (x + 3) & ~3; };
  long long best = -1, unsplit = -1;
  int best_n = 1;
  for (int n : cands) {
    if (n > s_max) break;
    int c = up4((P + n - 1) / n);
    c = std::max(std::max(c, kMinChunkPages), 4);
    int k = std::min(std::max(1, (P + c - 1) / c), s_max);  // splits of a P-page sequence
    const int per = up4((P + k - 1) / k);
    k = (P + per - 1) / per;
    const long long items = (long long)B * Hkv * k;
    const long long cost = (items + target_ctas - 1) / target_ctas * (c + 4) + (n > 1 ? 23 : 0);
    if (n == 1) unsplit = cost;
    if (best < 0 || cost < best) {
      best = cost;
      best_n = k;
    }
  }
  // (23 pages: the split's fixed cost, fitted when the merge was a second
  // launch; measured then: tiny decode 11.0 -> 6.0 us unsplit, ctx 512 x
  // B1 / B2 -11 / -20 %)
  if (best_n > 1 && best * 100 <= unsplit * 97) return true;
  const long long streams = (long long)B * Hkv;
  const long long rounds = (streams + target_ctas - 1) / target_ctas;
  const long long share = (streams * P + target_ctas - 1) / target_ctas;
  return P >= 128 && rounds * target_ctas * 10 >= streams * 11 && rounds * P - share >= 32;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct SplitWorkspace {
  size_t off_nsplit, off_lse, off_o, total;
};

// Split workspace: a split-bookkeeping region of 8 bytes per (sequence, kv
// head) -- the decode kernel's arrival words, or the engine's split counts
// (int32, per sequence, or per (sequence, kv head) stream under tile-granular
// shares) -- then LSE partials [s_max, rows, Hq] and O partials
// [s_max, rows, Hq, D] (fp32), each 256-byte aligned.  Nothing in it has to
// start at any particular value.
SplitWorkspace split_workspace_layout(int B, int Hkv, long long rows, int Hq, int D, int s_max) {
  SplitWorkspace w{};
  if (s_max <= 1) return w;
  w.off_nsplit = 0;
  w.off_lse = align256((size_t)B * Hkv * 8);
  w.off_o = w.off_lse + align256((size_t)s_max * rows * Hq * 4);
  w.total = w.off_o + align256((size_t)s_max * rows * Hq * D * 4);
  return w;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

int decode_resident_ctas(int D, int dtype, int rmax) {
  static int cache[2][2][4] = {};
  const int di = D == 128 ? 1 : 0, ri = rmax == 1 ? 0 : rmax == 2 ? 1 : rmax == 8 ? 2 : 3;
  int& c = cache[di][dtype][ri];
  if (c == 0) {
    const int per_sm = std::max(1, decode_ctas_per_sm(D, dtype, rmax));
    c = per_sm * num_sms();
  }
  return c;
}

int check_cache(const pa_tensor4& t, const char* name) {
  if (t.ptr == nullptr) return fail(PA_ERR_INVALID_ARG, "%s.ptr is NULL", name);
  if (!aligned16(t.ptr)) return fail(PA_ERR_INVALID_ARG, "%s.ptr must be 16-byte aligned", name);
  if (!mult8(t.stride_b) || !mult8(t.stride_t) || !mult8(t.stride_h))
    return fail(PA_ERR_INVALID_ARG,
                "%s strides must be positive multiples of 8 elements (got %lld, %lld, %lld)", name,
                (long long)t.stride_b, (long long)t.stride_t, (long long)t.stride_h);
  return PA_OK;
}

int check_common(int dtype, int D, int Hq, int Hkv) {
  if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "dtype %d", dtype);
  if (D != 64 && D != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim %d (64 or 128)", D);
  if (Hq < 1 || Hkv < 1) return fail(PA_ERR_INVALID_ARG, "head counts must be >= 1");
  if (Hq % Hkv != 0) return fail(PA_ERR_UNSUPPORTED, "Hq %d not a multiple of Hkv %d", Hq, Hkv);
  return PA_OK;
}

int rows_template(int rows) {
  return rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 8 ? 8 : 16;
}

}  // namespace

int set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int num_sms() {
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    sms[dev] = n;
  }
  return sms[dev];
}

bool encode_map(CUtensorMap* map, const void* base, int dtype, int D, int H, int64_t dim2,
                int64_t dim3, int64_t stride_h, int64_t stride_t, int64_t stride_b, int box_d,
                int box_h, int box_rows, bool swz = true) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)dim2, (cuuint64_t)dim3};
  const cuuint64_t strides[3] = {(cuuint64_t)stride_h * 2, (cuuint64_t)stride_t * 2,
                                 (cuuint64_t)stride_b * 2};
  const cuuint32_t box[4] = {(cuuint32_t)box_d, (cuuint32_t)box_h, (cuuint32_t)box_rows, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  // swz: 128-byte swizzle (64-column boxes for the tensor cores); the
  // CUDA-core decode reads unswizzled full-row boxes.
  const CUresult r = fn(map, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_cache_map(CUtensorMap* map, const void* base, int dtype, int D, int Hkv, int64_t dim2,
                      int64_t dim3, int64_t stride_h, int64_t stride_t, int64_t stride_b,
                      int box_d, int box_rows, bool swizzle128) {
  return encode_map(map, base, dtype, D, Hkv, dim2, dim3, stride_h, stride_t, stride_b, box_d, 1,
                    box_rows, swizzle128);
}

}  // namespace pa

using namespace pa;

// Rotary embedding applied inside the decode kernel (query blocks of up to
// kCudaCoreRows rows per kv head): tables, dimensions, pairing.
struct RopeArgs {
  const void* cos;
  const void* sin;
  int len, dim, interleaved;
};

static int fwd_kvcache_impl(const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                            pa_tensor4 k_cache, pa_tensor4 v_cache, const void* k_new,
                            const void* v_new, int Lnew, const int32_t* cache_seqlens,
                            const int32_t* block_table, int64_t bt_stride, int max_pages,
                            int page_size, int B, int Lq, int Hq, int Hkv, int D,
                            int64_t cache_extent, int max_seqlen_k, float scale, int causal,
                            int num_splits, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, int32_t* err_word, int dtype,
                            pa_stream_t stream, const RopeArgs* rope);

// Whether pa_fwd_kvcache_rotary rotates inside the attention launch (no
// scratch, no extra kernel): query blocks the decode kernel runs.
static bool rotary_fused(int Lq, int Hq, int Hkv) {
  return Hkv > 0 && Hq % Hkv == 0 && Lq * (Hq / Hkv) <= kCudaCoreRows;
}

extern "C" {

PA_API const char* pa_last_error_string(void) { return g_last_error.c_str(); }

PA_API int pa_version(void) { return 100; }

PA_API int pa_append_kv(pa_tensor4 k_cache, pa_tensor4 v_cache, const void* k_new,
                        const void* v_new, const int32_t* cache_seqlens,
                        const int32_t* block_table, int64_t bt_stride, int max_pages,
                        int page_size, int B, int Lnew, int Hkv, int D, int64_t cache_extent,
                        int dtype, int32_t* err_word, pa_stream_t stream) {
  int rc = check_common(dtype, D, Hkv, Hkv);
  if (rc) return rc;
  if (B < 0 || Lnew < 0) return fail(PA_ERR_INVALID_ARG, "negative B or Lnew");
  if (B == 0 || Lnew == 0) return PA_OK;
  if ((rc = check_cache(k_cache, "k_cache")) || (rc = check_cache(v_cache, "v_cache"))) return rc;
  if (k_new == nullptr || v_new == nullptr || cache_seqlens == nullptr)
    return fail(PA_ERR_INVALID_ARG, "k_new, v_new and cache_seqlens must be non-NULL");
  if (!aligned16(k_new) || !aligned16(v_new))
    return fail(PA_ERR_INVALID_ARG, "k_new/v_new must be 16-byte aligned");
  if (cache_extent < 1) return fail(PA_ERR_INVALID_ARG, "cache_extent must be >= 1");
  if (block_table != nullptr && (max_pages < 1 || bt_stride < max_pages))
    return fail(PA_ERR_INVALID_ARG, "block table needs max_pages >= 1 and bt_stride >= max_pages");
  int shift = 0;
  if (block_table != nullptr && !page_shift_of(page_size, &shift))
    return fail(PA_ERR_UNSUPPORTED, "page_size must be 16, 32, 64, 128 or 256");
  AppendParams p{};
  p.page_shift = shift;
  p.k_cache = k_cache.ptr;
  p.v_cache = v_cache.ptr;
  p.k_sb = k_cache.stride_b; p.k_st = k_cache.stride_t; p.k_sh = k_cache.stride_h;
  p.v_sb = v_cache.stride_b; p.v_st = v_cache.stride_t; p.v_sh = v_cache.stride_h;
  p.k_new = k_new;
  p.v_new = v_new;
  p.cache_seqlens = cache_seqlens;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.max_pages = max_pages;
  p.extent = cache_extent;
  p.B = B; p.Lnew = Lnew; p.Hkv = Hkv; p.D = D;
  p.err = err_word;
  const cudaError_t e = launch_append(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "append launch");
  return PA_OK;
}

PA_API size_t pa_fwd_kvcache_workspace_size(int B, int Lq, int Hq, int Hkv, int D,
                                            int max_seqlen_k, int num_splits) {
  if (B <= 0 || Lq <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return 0;
  const int G = Hq / Hkv;
  const int rows = Lq * G;
  // split partials exist for the CUDA-core decode and for packed engine items;
  // 128-row tiles of one head are never split
  if (rows > kEngineMaxRows || (rows > kCudaCoreRows && kEngineMaxRows % G != 0)) return 0;
  const int s_max = plan_s_max(B, Hkv, max_seqlen_k, num_splits);
  return split_workspace_layout(B, Hkv, (long long)B * Lq, Hq, D, s_max).total;
}

// scratch for the rotated q and k_new, ahead of pa_fwd_kvcache's own workspace
static size_t rotary_scratch_bytes(int B, int Lq, int Hq, int Hkv, int D, int Lnew) {
  const size_t qb = ((size_t)B * Lq * Hq * D * 2 + 255) & ~(size_t)255;
  const size_t kb = ((size_t)B * Lnew * Hkv * D * 2 + 255) & ~(size_t)255;
  return qb + kb;
}

PA_API size_t pa_fwd_kvcache_rotary_workspace_size(int B, int Lq, int Hq, int Hkv, int D, int Lnew,
                                                   int max_seqlen_k, int num_splits) {
  if (B <= 0 || Lq <= 0 || Lnew <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0) return 0;
  if (rotary_fused(Lq, Hq, Hkv))
    return pa_fwd_kvcache_workspace_size(B, Lq, Hq, Hkv, D, max_seqlen_k, num_splits);
  return rotary_scratch_bytes(B, Lq, Hq, Hkv, D, Lnew) +
         pa_fwd_kvcache_workspace_size(B, Lq, Hq, Hkv, D, max_seqlen_k, num_splits);
}

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
                                 int dtype, pa_stream_t stream) {
  int rc = check_common(dtype, D, Hq, Hkv);
  if (rc) return rc;
  if (B < 0 || Lq < 0) return fail(PA_ERR_INVALID_ARG, "negative B or Lq");
  if (B == 0 || Lq == 0) return PA_OK;
  if (Lnew < 1 || k_new == nullptr || v_new == nullptr || cache_seqlens == nullptr)
    return fail(PA_ERR_INVALID_ARG,
                "rotary embedding applies to appended tokens: needs Lnew >= 1, k_new, v_new and "
                "cache_seqlens");
  if (q == nullptr || rotary_cos == nullptr || rotary_sin == nullptr)
    return fail(PA_ERR_INVALID_ARG, "q, rotary_cos and rotary_sin must be non-NULL");
  if (rotary_dim < 2 || rotary_dim > D || rotary_dim % 2 != 0 || rotary_len < 1)
    return fail(PA_ERR_INVALID_ARG, "rotary_dim must be even in [2, D] and rotary_len >= 1");
  if (rotary_fused(Lq, Hq, Hkv)) {
    // the decode kernel rotates q as it stages it and k_new where it appends it
    const RopeArgs rope{rotary_cos, rotary_sin, rotary_len, rotary_dim, rotary_interleaved ? 1 : 0};
    return fwd_kvcache_impl(q, q_sb, q_st, q_sh, k_cache, v_cache, k_new, v_new, Lnew,
                            cache_seqlens, block_table, bt_stride, max_pages, page_size, B, Lq, Hq,
                            Hkv, D, cache_extent, max_seqlen_k, scale, causal, num_splits, out, lse,
                            workspace, workspace_bytes, err_word, dtype, stream, &rope);
  }
  const size_t scratch = rotary_scratch_bytes(B, Lq, Hq, Hkv, D, Lnew);
  if (workspace == nullptr || workspace_bytes < scratch ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(PA_ERR_WORKSPACE,
                "workspace must be 256-byte aligned and hold "
                "pa_fwd_kvcache_rotary_workspace_size bytes");
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  const size_t qb = ((size_t)B * Lq * Hq * D * 2 + 255) & ~(size_t)255;
  RotaryParams rp{};
  rp.q = q;
  rp.q_sb = q_sb; rp.q_st = q_st; rp.q_sh = q_sh;
  rp.k_new = k_new;
  rp.q_out = ws;
  rp.k_out = ws + qb;
  rp.cos = rotary_cos;
  rp.sin = rotary_sin;
  rp.cache_seqlens = cache_seqlens;
  rp.B = B; rp.Lq = Lq; rp.Lnew = Lnew; rp.Hq = Hq; rp.Hkv = Hkv; rp.D = D;
  rp.rotary_dim = rotary_dim;
  rp.rotary_len = rotary_len;
  rp.interleaved = rotary_interleaved ? 1 : 0;
  rp.err = err_word;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_rotary(rp, dtype, st);
  if (e != cudaSuccess) return cuda_fail(e, "rotary launch");
  const size_t rest = workspace_bytes - scratch;
  return pa_fwd_kvcache(ws, (int64_t)Lq * Hq * D, (int64_t)Hq * D, D, k_cache, v_cache, ws + qb,
                        v_new, Lnew, cache_seqlens, block_table, bt_stride, max_pages, page_size,
                        B, Lq, Hq, Hkv, D, cache_extent, max_seqlen_k, scale, causal, num_splits,
                        out, lse,
                        rest ? ws + scratch : nullptr, rest, err_word, dtype, stream);
}

PA_API size_t pa_fwd_varlen_workspace_size(int B, int total_q, int max_seqlen_q, int Hq,
                                           int Hkv, int D, int max_seqlen_k) {
  if (B <= 0 || total_q <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return 0;
  (void)max_seqlen_q;
  const int s_max = plan_s_max(std::min(B, kDecodeMaxSchedB), Hkv, max_seqlen_k, 0);
  return split_workspace_layout(B, Hkv, total_q, Hq, D, s_max).total;
}

PA_API int pa_fwd_kvcache(const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                          pa_tensor4 k_cache, pa_tensor4 v_cache, const void* k_new,
                          const void* v_new, int Lnew, const int32_t* cache_seqlens,
                          const int32_t* block_table, int64_t bt_stride, int max_pages,
                          int page_size, int B, int Lq, int Hq, int Hkv, int D,
                          int64_t cache_extent, int max_seqlen_k,
                          float scale, int causal, int num_splits, void* out, float* lse,
                          void* workspace, size_t workspace_bytes, int32_t* err_word, int dtype,
                          pa_stream_t stream) {
  return fwd_kvcache_impl(q, q_sb, q_st, q_sh, k_cache, v_cache, k_new, v_new, Lnew,
                          cache_seqlens, block_table, bt_stride, max_pages, page_size, B, Lq, Hq,
                          Hkv, D, cache_extent, max_seqlen_k, scale, causal, num_splits, out, lse,
                          workspace, workspace_bytes, err_word, dtype, stream, nullptr);
}

}  // extern "C"

static int fwd_kvcache_impl(const void* q, int64_t q_sb, int64_t q_st, int64_t q_sh,
                            pa_tensor4 k_cache, pa_tensor4 v_cache, const void* k_new,
                            const void* v_new, int Lnew, const int32_t* cache_seqlens,
                            const int32_t* block_table, int64_t bt_stride, int max_pages,
                            int page_size, int B, int Lq, int Hq, int Hkv, int D,
                            int64_t cache_extent, int max_seqlen_k, float scale, int causal,
                            int num_splits, void* out, float* lse, void* workspace,
                            size_t workspace_bytes, int32_t* err_word, int dtype,
                            pa_stream_t stream, const RopeArgs* rope) {
  int rc = check_common(dtype, D, Hq, Hkv);
  if (rc) return rc;
  if (B < 0 || Lq < 0 || Lnew < 0 || max_seqlen_k < 0 || num_splits < 0)
    return fail(PA_ERR_INVALID_ARG, "negative size argument");
  if (B == 0) return PA_OK;
  if ((rc = check_cache(k_cache, "k_cache")) || (rc = check_cache(v_cache, "v_cache"))) return rc;
  if (cache_seqlens == nullptr) return fail(PA_ERR_INVALID_ARG, "cache_seqlens is NULL");
  if (Lnew > 0 && (k_new == nullptr || v_new == nullptr || !aligned16(k_new) || !aligned16(v_new)))
    return fail(PA_ERR_INVALID_ARG, "Lnew > 0 needs 16-byte aligned k_new and v_new");
  if (cache_extent < 1) return fail(PA_ERR_INVALID_ARG, "cache_extent must be >= 1");
  if (block_table != nullptr && (max_pages < 1 || bt_stride < max_pages))
    return fail(PA_ERR_INVALID_ARG, "block table needs max_pages >= 1 and bt_stride >= max_pages");
  int shift = 0;
  if (block_table != nullptr && !page_shift_of(page_size, &shift))
    return fail(PA_ERR_UNSUPPORTED, "page_size must be 16, 32, 64, 128 or 256");
  const int64_t page_rows = (int64_t)kPage << shift;
  if (Lq == 0) {
    if (Lnew == 0) return PA_OK;
    return pa_append_kv(k_cache, v_cache, k_new, v_new, cache_seqlens, block_table, bt_stride,
                        max_pages, page_size, B, Lnew, Hkv, D, cache_extent, dtype, err_word,
                        stream);
  }
  if (q == nullptr || out == nullptr) return fail(PA_ERR_INVALID_ARG, "q and out must be non-NULL");
  if (!aligned16(q) || !aligned16(out))
    return fail(PA_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
  if (!mult8(q_sh) || !mult8(q_st) || !mult8(q_sb))
    return fail(PA_ERR_INVALID_ARG, "q strides must be positive multiples of 8 elements");
  if (!(scale > 0.f) || !std::isfinite(scale))
    return fail(PA_ERR_INVALID_ARG, "scale must be finite and > 0");

  const int G = Hq / Hkv;
  const int rows = Lq * G;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (rope != nullptr && (rows > kCudaCoreRows || Lnew < 1))
    return fail(PA_ERR_INVALID_ARG, "in-kernel rotary embedding needs an append and <= %d rows",
                kCudaCoreRows);
  if (rows > kCudaCoreRows) {
    // Tensor-core engine: the new tokens are appended first (same stream),
    // then every key is read from the cache.  Query blocks of up to 128 rows
    // per kv head run packed (all G heads of a kv head in one tile, split-KV);
    // longer ones as 128-row tiles of one head.
    if (Lnew > 0) {
      rc = pa_append_kv(k_cache, v_cache, k_new, v_new, cache_seqlens, block_table, bt_stride,
                        max_pages, page_size, B, Lnew, Hkv, D, cache_extent, dtype, err_word,
                        stream);
      if (rc) return rc;
    }
    const bool pack = rows <= kEngineMaxRows && (kEngineMaxRows % G) == 0;
    const int s_max = pack ? plan_s_max(B, Hkv, max_seqlen_k, num_splits) : 1;
    const SplitWorkspace ws = split_workspace_layout(B, Hkv, (long long)B * Lq, Hq, D, s_max);
    if (ws.total > 0 && (workspace == nullptr || workspace_bytes < ws.total))
      return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", ws.total,
                  workspace_bytes);
    const bool paged_p = block_table != nullptr;
    CUtensorMap tq1, tq2, tk, tv;
    if (!encode_map(&tq1, q, dtype, D, Hq, Lq, B, q_sh, q_st, q_sb, 64, 1, 128) ||
        !encode_map(&tq2, q, dtype, D, Hq, Lq, B, q_sh, q_st, q_sb, 64, pack ? G : 1,
                    pack ? kEngineMaxRows / G : 128) ||
        !encode_map(&tk, k_cache.ptr, dtype, D, Hkv, paged_p ? page_rows : cache_extent,
                    paged_p ? cache_extent : B, k_cache.stride_h, k_cache.stride_t,
                    k_cache.stride_b, 64, 1, kPage) ||
        !encode_map(&tv, v_cache.ptr, dtype, D, Hkv, paged_p ? page_rows : cache_extent,
                    paged_p ? cache_extent : B, v_cache.stride_h, v_cache.stride_t,
                    v_cache.stride_b, 64, 1, kPage))
      return fail(PA_ERR_INVALID_ARG, "cannot encode a TMA descriptor for q or the caches");
    const int grid = engine_grid();
    EngineParams ep{};
    ep.out = out;
    ep.lse = lse;
    ep.cache_seqlens = cache_seqlens;
    ep.Lnew = Lnew;
    ep.block_table = block_table;
    ep.bt_stride = bt_stride;
    ep.max_pages = paged_p ? max_pages : 0;
    ep.page_shift = shift;
    ep.extent = cache_extent;
    ep.B = B; ep.Lq = Lq; ep.Hq = Hq; ep.Hkv = Hkv; ep.G = G;
    ep.max_seqlen_k = max_seqlen_k;
    ep.total_q = 0;
    ep.pack_rows = pack ? kEngineMaxRows : 0;
    ep.max_q_tiles = (Lq + kEngineMaxRows - 1) / kEngineMaxRows;
    ep.scale_log2 = scale * kLog2e;
    ep.causal = causal ? 1 : 0;
    ep.s_max = s_max;
    ep.target_ctas = num_splits > 0 ? (1 << 30) : 2 * grid;
    ep.min_chunk_pages = num_splits > 0 ? 1 : kMinChunkPages;
    // automatic splits of packed items: tile-granular shares, split counts per
    // (sequence, kv head) stream
    ep.tilebal = (pack && s_max > 1 && num_splits == 0) ? 1 : 0;
    uint8_t* wsb = reinterpret_cast<uint8_t*>(workspace);
    ep.nsplit = ws.total ? reinterpret_cast<int32_t*>(wsb + ws.off_nsplit) : nullptr;
    ep.lse_part = ws.total ? reinterpret_cast<float*>(wsb + ws.off_lse) : nullptr;
    ep.o_part = ws.total ? reinterpret_cast<float*>(wsb + ws.off_o) : nullptr;
    ep.err = err_word;
    // query blocks longer than one packed tile: two 128-row query tiles per
    // CTA sharing every K/V tile; packed blocks (decode, multi-query decode):
    // the engine, split over the keys
    cudaError_t e = pack ? launch_engine(ep, tq1, tq2, tk, tv, D, dtype, grid, st)
                         : launch_prefill(ep, tq1, tk, tv, D, dtype, st);
    if (e != cudaSuccess) return cuda_fail(e, pack ? "engine launch" : "prefill launch");
    if (s_max > 1) {
      CombineParams c{};
      c.o_part = ep.o_part;
      c.lse_part = ep.lse_part;
      c.nsplit = ep.nsplit;
      c.ns_stride = ep.tilebal ? Hkv : 1;  // counts per stream, or per sequence
      c.ns_group = ep.tilebal ? G : Hq;
      c.S = s_max;
      c.B = B; c.Lq = Lq; c.Hq = Hq;
      c.cu_seqlens_q = nullptr;
      c.total_q = 0;
      c.out = out;
      c.lse = lse;
      e = launch_combine(c, D, dtype, B * Lq, st, true);
      if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    }
    return PA_OK;
  }

  const int rmax = rows_template(rows);
  const int resident = decode_resident_ctas(D, dtype, rmax);
  int s_max = plan_s_max(B, Hkv, max_seqlen_k, num_splits);
  if (num_splits == 0 && !decode_splits_useful(B, Hkv, max_seqlen_k, s_max, resident)) s_max = 1;
  const SplitWorkspace ws = split_workspace_layout(B, Hkv, (long long)B * Lq, Hq, D, s_max);
  if (ws.total > 0 && (workspace == nullptr || workspace_bytes < ws.total))
    return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", ws.total,
                workspace_bytes);

  CUtensorMap tmk, tmv;
  const bool paged = block_table != nullptr;
  const int64_t dim2 = paged ? page_rows : cache_extent;
  const int64_t dim3 = paged ? cache_extent : B;
  // 1-2 rows: full-row unswizzled page boxes; more: 64-column boxes with the
  // 128-byte swizzle that the tensor-core consumer's ldmatrix reads
  const bool swz = rmax > 2;
  if (!encode_cache_map(&tmk, k_cache.ptr, dtype, D, Hkv, dim2, dim3, k_cache.stride_h,
                        k_cache.stride_t, k_cache.stride_b, swz ? 64 : D, kPage, swz) ||
      !encode_cache_map(&tmv, v_cache.ptr, dtype, D, Hkv, dim2, dim3, v_cache.stride_h,
                        v_cache.stride_t, v_cache.stride_b, swz ? 64 : D, kPage, swz))
    return fail(PA_ERR_INVALID_ARG, "cannot encode a TMA descriptor for the cache views");

  DecodeParams p{};
  p.q = q;
  p.q_sb = q_sb; p.q_st = q_st; p.q_sh = q_sh;
  p.out = out;
  p.lse = lse;
  p.k_new = k_new;
  p.v_new = v_new;
  p.Lnew = Lnew;
  p.k_cache = k_cache.ptr;
  p.v_cache = v_cache.ptr;
  p.k_sb = k_cache.stride_b; p.k_st = k_cache.stride_t; p.k_sh = k_cache.stride_h;
  p.v_sb = v_cache.stride_b; p.v_st = v_cache.stride_t; p.v_sh = v_cache.stride_h;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.max_pages = paged ? max_pages : 0;
  p.page_shift = shift;
  p.extent = cache_extent;
  p.cache_seqlens = cache_seqlens;
  p.B = B; p.Lq = Lq; p.Hq = Hq; p.Hkv = Hkv; p.G = G;
  p.max_seqlen_k = max_seqlen_k;
  p.scale_log2 = scale * kLog2e;
  p.causal = causal ? 1 : 0;
  p.s_max = s_max;
  p.target_ctas = num_splits > 0 ? (1 << 30) : resident;
  p.grid_ctas = resident;
  p.min_chunk_pages = num_splits > 0 ? 1 : kMinChunkPages;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(workspace);
  p.split_ctr = ws.total ? reinterpret_cast<unsigned long long*>(wsb + ws.off_nsplit) : nullptr;
  p.lse_part = ws.total ? reinterpret_cast<float*>(wsb + ws.off_lse) : nullptr;
  p.o_part = ws.total ? reinterpret_cast<float*>(wsb + ws.off_o) : nullptr;
  p.err = err_word;
  if (rope != nullptr) {
    p.rot_cos = rope->cos;
    p.rot_sin = rope->sin;
    p.rot_len = rope->len;
    p.rot_dim = rope->dim;
    p.rot_interleaved = rope->interleaved;
  }

  // one launch: the last split of every stream to finish merges the stream
  const cudaError_t e = launch_decode(p, tmk, tmv, D, dtype, rmax, st);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return PA_OK;
}

extern "C" {

PA_API int pa_fwd_varlen_unified(const void* q, int64_t q_st, int64_t q_sh, pa_tensor4 k_cache,
                                 pa_tensor4 v_cache, const int32_t* cu_seqlens_q,
                                 const int32_t* seqlens_k, const int32_t* block_table,
                                 int64_t bt_stride, int max_pages, int page_size, int B,
                                 int total_q,
                                 int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D,
                                 int64_t num_pages, float scale, int causal, void* out,
                                 float* lse, void* workspace, size_t workspace_bytes,
                                 int32_t* err_word, int dtype, pa_stream_t stream) {
  int rc = check_common(dtype, D, Hq, Hkv);
  if (rc) return rc;
  if (B < 0 || total_q < 0 || max_seqlen_q < 0 || max_seqlen_k < 0)
    return fail(PA_ERR_INVALID_ARG, "negative size argument");
  if (B == 0 || total_q == 0) return PA_OK;
  if ((rc = check_cache(k_cache, "k_cache")) || (rc = check_cache(v_cache, "v_cache"))) return rc;
  if (q == nullptr || out == nullptr || cu_seqlens_q == nullptr || seqlens_k == nullptr ||
      block_table == nullptr)
    return fail(PA_ERR_INVALID_ARG, "q, out, cu_seqlens_q, seqlens_k, block_table must be non-NULL");
  if (!aligned16(q) || !aligned16(out)) return fail(PA_ERR_INVALID_ARG, "q/out 16-byte alignment");
  if (!mult8(q_st) || !mult8(q_sh)) return fail(PA_ERR_INVALID_ARG, "q strides multiples of 8");
  if (max_pages < 1 || bt_stride < max_pages || num_pages < 1)
    return fail(PA_ERR_INVALID_ARG, "block table / pool sizes");
  int shift = 0;
  if (!page_shift_of(page_size, &shift))
    return fail(PA_ERR_UNSUPPORTED, "page_size must be 16, 32, 64, 128 or 256");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(PA_ERR_INVALID_ARG, "scale");
  if (B > kEngineMaxB) return fail(PA_ERR_UNSUPPORTED, "more than %d sequences", kEngineMaxB);
  const int G = Hq / Hkv;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // One engine launch over the whole mixed batch: sequences of up to 128
  // query rows per kv head (decode, multi-query decode, short chunks) run as
  // packed split-KV items, longer chunks as 128-row tiles of one head.
  const bool pack = (kEngineMaxRows % G) == 0;
  const int s_max = pack ? plan_s_max(B, Hkv, max_seqlen_k, 0) : 1;
  const SplitWorkspace ws = split_workspace_layout(B, Hkv, total_q, Hq, D, s_max);
  if (ws.total > 0 && (workspace == nullptr || workspace_bytes < ws.total))
    return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes required (got %zu)", ws.total,
                workspace_bytes);
  CUtensorMap tq1, tq2, tk, tv;
  if (!encode_map(&tq1, q, dtype, D, Hq, total_q, 1, q_sh, q_st, q_st * total_q, 64, 1, 128) ||
      !encode_map(&tq2, q, dtype, D, Hq, total_q, 1, q_sh, q_st, q_st * total_q, 64,
                  pack ? G : 1, pack ? kEngineMaxRows / G : 128) ||
      !encode_map(&tk, k_cache.ptr, dtype, D, Hkv, page_size, num_pages, k_cache.stride_h,
                  k_cache.stride_t, k_cache.stride_b, 64, 1, kPage) ||
      !encode_map(&tv, v_cache.ptr, dtype, D, Hkv, page_size, num_pages, v_cache.stride_h,
                  v_cache.stride_t, v_cache.stride_b, 64, 1, kPage))
    return fail(PA_ERR_INVALID_ARG, "cannot encode a TMA descriptor for q or the caches");
  const int grid = engine_grid();
  EngineParams ep{};
  ep.out = out;
  ep.lse = lse;
  ep.cu_seqlens_q = cu_seqlens_q;
  ep.seqlens_k = seqlens_k;
  ep.block_table = block_table;
  ep.bt_stride = bt_stride;
  ep.max_pages = max_pages;
  ep.page_shift = shift;
  ep.extent = num_pages;
  ep.B = B; ep.Lq = 0; ep.Hq = Hq; ep.Hkv = Hkv; ep.G = G;
  ep.max_seqlen_k = max_seqlen_k;
  ep.total_q = total_q;
  ep.pack_rows = pack ? kEngineMaxRows : 0;
  ep.max_q_tiles = (max_seqlen_q + kEngineMaxRows - 1) / kEngineMaxRows;
  ep.scale_log2 = scale * kLog2e;
  ep.causal = causal ? 1 : 0;
  ep.s_max = s_max;
  ep.target_ctas = 2 * grid;
  ep.min_chunk_pages = kMinChunkPages;
  uint8_t* wsb = reinterpret_cast<uint8_t*>(workspace);
  ep.nsplit = ws.total ? reinterpret_cast<int32_t*>(wsb + ws.off_nsplit) : nullptr;
  ep.lse_part = ws.total ? reinterpret_cast<float*>(wsb + ws.off_lse) : nullptr;
  ep.o_part = ws.total ? reinterpret_cast<float*>(wsb + ws.off_o) : nullptr;
  ep.err = err_word;
  cudaError_t e = launch_engine(ep, tq1, tq2, tk, tv, D, dtype, grid, st);
  if (e != cudaSuccess) return cuda_fail(e, "engine launch");
  if (s_max > 1) {
    CombineParams c{};
    c.o_part = ep.o_part;
    c.lse_part = ep.lse_part;
    c.nsplit = ep.nsplit;
    c.ns_stride = 1;
    c.ns_group = Hq;
    c.S = s_max;
    c.B = B; c.Lq = 0; c.Hq = Hq;
    c.cu_seqlens_q = cu_seqlens_q;
    c.total_q = total_q;
    c.out = out;
    c.lse = lse;
    e = launch_combine(c, D, dtype, total_q, st, true);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  }
  return PA_OK;
}


PA_API int pa_split_combine(const float* o_partial, const float* lse_partial,
                            const int32_t* splits_per_seq, int S, int B, int Lq, int Hq, int D,
                            void* out, float* lse, int dtype, pa_stream_t stream) {
  if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "dtype %d", dtype);
  if (D != 64 && D != 128) return fail(PA_ERR_UNSUPPORTED, "head_dim %d", D);
  if (S < 1 || B < 0 || Lq < 0 || Hq < 1) return fail(PA_ERR_INVALID_ARG, "sizes");
  if (B == 0 || Lq == 0) return PA_OK;
  if (o_partial == nullptr || lse_partial == nullptr || out == nullptr)
    return fail(PA_ERR_INVALID_ARG, "o_partial, lse_partial and out must be non-NULL");
  if (!aligned16(o_partial) || !aligned16(out))
    return fail(PA_ERR_INVALID_ARG, "o_partial/out must be 16-byte aligned");
  CombineParams c{};
  c.o_part = o_partial;
  c.lse_part = lse_partial;
  c.nsplit = splits_per_seq;
  c.ns_stride = 1;
  c.ns_group = Hq;
  c.S = S;
  c.B = B; c.Lq = Lq; c.Hq = Hq;
  c.cu_seqlens_q = nullptr;
  c.total_q = 0;
  c.out = out;
  c.lse = lse;
  const cudaError_t e =
      launch_combine(c, D, dtype, B * Lq, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  return PA_OK;
}

}  // extern "C"
