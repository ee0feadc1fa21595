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

constexpr int kCombineWarps = 8;

template <int D, typename T>
__global__ void __launch_bounds__(kCombineWarps * 32)
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
    const int n = p.nsplit ? min(__ldg(p.nsplit + b), p.S) : p.S;
    if (n <= 0) continue;
    // max of the split LSEs (natural log) -> log2 domain; lane s keeps the
    // LSE of split s (and of s + 32, ...)
    float M = neg_inf();
    float my_ls = neg_inf();
    for (int s = lane; s < n; s += 32) {
      const float ls = __ldg(p.lse_part + ((long long)s * NR + row) * p.Hq + h) * kLog2e;
      if (s == lane) my_ls = ls;
      M = fmaxf(M, ls);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float acc[kPVE];
#pragma unroll
    for (int e = 0; e < kPVE; ++e) acc[e] = 0.f;
    float L = 0.f;
    if (M != neg_inf()) {
      // four splits per step: their partial rows are loaded together; an
      // empty split (LSE -inf) gets weight 0 and its partial is not read
      constexpr int kU = 4;
      for (int s0 = 0; s0 < n; s0 += kU) {
        float wgt[kU];
        float v[kU][kPVE];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int s = s0 + u;
          float ls = neg_inf();
          if (s < 32) {
            ls = __shfl_sync(0xffffffffu, my_ls, s & 31);
          } else if (s < n) {
            ls = __ldg(p.lse_part + ((long long)s * NR + row) * p.Hq + h) * kLog2e;
          }
          const bool live = s < n && ls != neg_inf();
          wgt[u] = live ? ex2(ls - M) : 0.f;
          const float* op = p.o_part + (((long long)s * NR + row) * p.Hq + h) * D + lane * kPVE;
#pragma unroll
          for (int e = 0; e < kPVE; ++e) v[u][e] = 0.f;
          if (live) {
            if constexpr (kPVE == 4) {
              const float4 x = __ldg(reinterpret_cast<const float4*>(op));
              v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
            } else {
              const float2 x = __ldg(reinterpret_cast<const float2*>(op));
              v[u][0] = x.x; v[u][1] = x.y;
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          L += wgt[u];
#pragma unroll
          for (int e = 0; e < kPVE; ++e) acc[e] = fmaf(wgt[u], v[u][e], acc[e]);
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
