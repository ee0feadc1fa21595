// Rotary position embedding of a kvcache call's new tokens (sm_103a): q at
// the positions of the new tokens and k_new at the slots the append writes
// them to, into scratch buffers that the attention path then reads in place
// of q and k_new.  The feature is named on flash-attention #824 "Add support
// for small page sizes" (a fix to fused RoPE embeddings in the kvcache
// forward); the rotation is the published RoFormer one (each feature pair
// rotated by pos * theta_p, cos / sin tables supplied by the caller), with the
// split-halves or interleaved pairing.
//
// One warp per (token, head) row; lanes take feature pairs.  The rotation is
// computed in fp32 -- for fp16 / bf16 inputs each product is exact in fp32,
// so y = fma(x1, c, -(x2 s)) is the exact x1 c - x2 s rounded once -- and
// rounded once to the storage type.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) rotary_kernel(const RotaryParams p) {
  using E = Elem<T>;
  const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const long long nq = (long long)p.B * p.Lq * p.Hq;
  const long long nk = (long long)p.B * p.Lnew * p.Hkv;
  if (row >= nq + nk) return;
  const T* src;
  T* dst;
  int b, pos;
  if (row < nq) {
    const int h = (int)(row % p.Hq);
    const int i = (int)((row / p.Hq) % p.Lq);
    b = (int)(row / ((long long)p.Hq * p.Lq));
    src = reinterpret_cast<const T*>(p.q) + b * p.q_sb + i * p.q_st + h * p.q_sh;
    dst = reinterpret_cast<T*>(p.q_out) + row * p.D;
    // query row i is the (Lnew - Lq + i)-th new token
    pos = __ldg(p.cache_seqlens + b) + p.Lnew - p.Lq + i;
  } else {
    const long long r = row - nq;
    const int i = (int)((r / p.Hkv) % p.Lnew);
    b = (int)(r / ((long long)p.Hkv * p.Lnew));
    src = reinterpret_cast<const T*>(p.k_new) + r * p.D;
    dst = reinterpret_cast<T*>(p.k_out) + r * p.D;
    pos = __ldg(p.cache_seqlens + b) + i;
  }
  const bool ok = pos >= 0 && pos < p.rotary_len;
  if (!ok && lane == 0) report(p.err, PA_DEVERR_LENGTH, b, pos);
  const int half = p.rotary_dim / 2;
  const T* cs = reinterpret_cast<const T*>(p.cos) + (long long)(ok ? pos : 0) * half;
  const T* sn = reinterpret_cast<const T*>(p.sin) + (long long)(ok ? pos : 0) * half;
  for (int q = lane; q < half; q += 32) {
    const int i1 = p.interleaved ? 2 * q : q;
    const int i2 = p.interleaved ? 2 * q + 1 : q + half;
    const float x1 = static_cast<float>(src[i1]);
    const float x2 = static_cast<float>(src[i2]);
    float y1 = x1, y2 = x2;
    if (ok) {
      const float c = static_cast<float>(cs[q]);
      const float s = static_cast<float>(sn[q]);
      y1 = fmaf(x1, c, -(x2 * s));
      y2 = fmaf(x1, s, x2 * c);
    }
    dst[i1] = E::from_f(y1);
    dst[i2] = E::from_f(y2);
  }
  for (int d = p.rotary_dim + lane; d < p.D; d += 32) dst[d] = src[d];
}

}  // namespace

cudaError_t launch_rotary(const RotaryParams& p, int dtype, cudaStream_t st) {
  const long long rows = (long long)p.B * p.Lq * p.Hq + (long long)p.B * p.Lnew * p.Hkv;
  if (rows == 0) return cudaSuccess;
  const long long blocks = (rows * 32 + 255) / 256;
  if (dtype == PA_F16)
    rotary_kernel<__half><<<(unsigned)blocks, 256, 0, st>>>(p);
  else
    rotary_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
