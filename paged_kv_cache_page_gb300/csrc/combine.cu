// Split-KV combine (sm_103a): merges per-split normalised outputs O_s and
// their log-sum-exps LSE_s into LSE = ln sum_s exp(LSE_s) and
// O = sum_s exp(LSE_s - LSE) O_s -- the step that follows a split-KV forward
// (vLLM #6052 "Unify the kernel used in flash attention backend", comment on
// flash_fwd_splitkv_kernel being chosen for num_splits == 0 with a page
// table).  One warp per (query row, head); lanes own D/32 columns, so every
// split row is read with one coalesced 128-bit (D = 128) or 64-bit access per
// lane.  The split weights are computed in the log2 domain.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Four warps per block: small enough (with the register cap below) to be
// resident beside a decode CTA, so the blocks of a programmatic dependent
// launch wait on the SMs rather than behind the decode grid.
constexpr int kCombineWarps = 4;

// At most 56 registers a thread (nine blocks' worth per SM): a 4-warp block
// then fits in the registers a 10-warp decode CTA of 168 leaves free.
template <int D, typename T>
__global__ void __launch_bounds__(kCombineWarps * 32, 9)
    combine_kernel(const CombineParams p, const long long rows_total) {
  using E = Elem<T>;
  constexpr int kPVE = D / 32;
  // partials are complete once the producing grid has finished (a no-op when
  // this launch does not depend on one programmatically)
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const long long w0 = (long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  const long long nwarps = (long long)gridDim.x * kCombineWarps;
  const long long NR = p.cu_seqlens_q ? (long long)p.total_q : (long long)p.B * p.Lq;
  for (long long w = w0; w < rows_total * p.Hq; w += nwarps) {
    const long long row = w / p.Hq;
    const int h = (int)(w % p.Hq);
    int b, qi;
    if (p.cu_seqlens_q != nullptr) {
      int lo = 0, hi = p.B;  // last b with cu[b] <= row
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.cu_seqlens_q + mid) <= row) lo = mid; else hi = mid;
      }
      b = lo;
      qi = (int)(row - __ldg(p.cu_seqlens_q + b));
    } else {
      b = (int)(row / p.Lq);
      qi = (int)(row % p.Lq);
    }
    // The split count, the LSE of split `lane` and the first kU partial
    // rows are loaded together (every index is below S, the splits the
    // partial arrays hold) and masked once the count is known: one round
    // trip to L2 instead of three dependent ones.
    constexpr int kU = kPVE == 4 ? 6 : 8;
    const long long base = (long long)row * p.Hq + h;    // (row, head) of split 0
    const long long sstride = NR * p.Hq;                 // one split further
    const int ns = p.nsplit ? __ldg(p.nsplit + (long long)b * p.ns_stride + h / p.ns_group) : p.S;
    const float ls_lane = lane < p.S ? __ldg(p.lse_part + lane * sstride + base) * kLog2e : neg_inf();
    float v0[kU][kPVE];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
#pragma unroll
      for (int e = 0; e < kPVE; ++e) v0[u][e] = 0.f;
      if (u < p.S) {
        const float* op = p.o_part + (u * sstride + base) * D + lane * kPVE;
        if constexpr (kPVE == 4) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(op));
          v0[u][0] = x.x; v0[u][1] = x.y; v0[u][2] = x.z; v0[u][3] = x.w;
        } else {
          const float2 x = __ldg(reinterpret_cast<const float2*>(op));
          v0[u][0] = x.x; v0[u][1] = x.y;
        }
      }
    }
    const int n = min(ns, p.S);
    if (n <= 0) continue;
    // max of the split LSEs (natural log -> log2 domain); lane s keeps the
    // LSE of split s < 32
    const float my_ls = lane < n ? ls_lane : neg_inf();
    float M = my_ls;
    for (int s = lane + 32; s < n; s += 32) M = fmaxf(M, __ldg(p.lse_part + s * sstride + base) * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[kPVE];
#pragma unroll
    for (int e = 0; e < kPVE; ++e) acc[e] = 0.f;
    float L = 0.f;
    if (M != neg_inf()) {
      // an empty split (LSE -inf) gets weight 0 and its partial row, which
      // may hold anything, is never used
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const float ls = __shfl_sync(0xffffffffu, my_ls, u);
        const bool live = u < n && ls != neg_inf();
        const float wgt = live ? ex2(ls - M) : 0.f;
        L += wgt;
#pragma unroll
        for (int e = 0; e < kPVE; ++e) acc[e] = live ? fmaf(wgt, v0[u][e], acc[e]) : acc[e];
      }
      for (int s = kU; s < n; ++s) {
        const float ls = s < 32 ? __shfl_sync(0xffffffffu, my_ls, s)
                                : __ldg(p.lse_part + s * sstride + base) * kLog2e;
        if (ls == neg_inf()) continue;
        const float wgt = ex2(ls - M);
        L += wgt;
        const float* op = p.o_part + (s * sstride + base) * D + lane * kPVE;
        if constexpr (kPVE == 4) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(op));
          acc[0] = fmaf(wgt, x.x, acc[0]);
          acc[1] = fmaf(wgt, x.y, acc[1]);
          acc[2] = fmaf(wgt, x.z, acc[2]);
          acc[3] = fmaf(wgt, x.w, acc[3]);
        } else {
          const float2 x = __ldg(reinterpret_cast<const float2*>(op));
          acc[0] = fmaf(wgt, x.x, acc[0]);
          acc[1] = fmaf(wgt, x.y, acc[1]);
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    T* orow = reinterpret_cast<T*>(p.out) + (row * p.Hq + h) * D + lane * kPVE;
    if constexpr (kPVE == 4) {
      uint2 u;
      u.x = E::from_f2(acc[0] * inv, acc[1] * inv);
      u.y = E::from_f2(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(orow) = u;
    } else {
      *reinterpret_cast<uint32_t*>(orow) = E::from_f2(acc[0] * inv, acc[1] * inv);
    }
    if (p.lse != nullptr && lane == 0) {
      const float lse_v = L > 0.f ? (M + lg2(L)) * kLn2 : neg_inf();
      if (p.cu_seqlens_q != nullptr)
        p.lse[(long long)h * p.total_q + row] = lse_v;
      else
        p.lse[((long long)b * p.Hq + h) * p.Lq + qi] = lse_v;
    }
  }
}

template <int D, typename T>
cudaError_t launch_t(const CombineParams& p, long long rows_total, cudaStream_t st,
                     bool dependent) {
  if (p.nsplit != nullptr && (p.ns_stride < 1 || p.ns_group < 1)) return cudaErrorInvalidValue;
  // the shared-memory carveout the decode kernels run with, so that waiting
  // blocks can share their SMs
  static bool carveout_set = false;
  if (!carveout_set) {
    const cudaError_t e = cudaFuncSetAttribute(
        combine_kernel<D, T>, cudaFuncAttributePreferredSharedMemoryCarveout,
        (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    carveout_set = true;
  }
  const long long warps = rows_total * p.Hq;
  long long blocks = (warps + kCombineWarps - 1) / kCombineWarps;
  const long long cap = 152LL * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel<D, T>, p, rows_total);
}

}  // namespace

cudaError_t launch_combine(const CombineParams& p, int D, int dtype, int rows_total,
                           cudaStream_t st, bool dependent) {
  if (D == 128 && dtype == PA_F16) return launch_t<128, __half>(p, rows_total, st, dependent);
  if (D == 128 && dtype == PA_BF16)
    return launch_t<128, __nv_bfloat16>(p, rows_total, st, dependent);
  if (D == 64 && dtype == PA_F16) return launch_t<64, __half>(p, rows_total, st, dependent);
  if (D == 64 && dtype == PA_BF16)
    return launch_t<64, __nv_bfloat16>(p, rows_total, st, dependent);
  return cudaErrorInvalidValue;
}

}  // namespace pa
