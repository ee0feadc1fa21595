// Tensor-core rate of the attention MMA shapes (test-only library): every CTA
// (one per SM) issues `n_instr` back-to-back kind::f16 MMAs of M = 128,
// K = 16 and N in {128, 256} into one TMEM accumulator, A from shared memory
// or from TMEM, and its first thread times issue and completion with the SM
// clock.  `ksteps` = 4 cycles through the four 16-element k-steps of one
// 128-byte slab (operands repeat every 4 instructions); 8 walks two slabs, so
// every instruction of a K = 128 product reads distinct operand bytes, as the
// attention tiles do.  Attention with head dim 128 runs Q K^T at N = 128 keys per tile and
// P V at N = D = 128; this measures what that shape can reach on the hardware,
// next to the N = 256 shape a plain GEMM uses.
#include <cuda_runtime.h>

#include "pa_common.cuh"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kRateSmem = 120 * 1024;  // one CTA per SM

__global__ void __launch_bounds__(128, 1)
    mma_rate_kernel(int n_instr, int N, int a_in_tmem, int ksteps, long long* cycles) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;          // two slabs of 128 rows x 128 bytes, 128-byte swizzle
  uint8_t* sB = smem + 32768;  // two slabs of N rows x 128 bytes
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 32768 + 65536);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + 32768 + 65536 + 64);
  const int tid = threadIdx.x, warp = tid >> 5;
  // operands: fp16 1.0 everywhere (values do not matter for the rate)
  for (int i = tid; i < (32768 + 65536) / 16; i += 128)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0x3c003c00u, 0x3c003c00u, 0x3c003c00u,
                                                   0x3c003c00u);
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tc::tmem_alloc(tslot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  // A in TMEM: columns [384, 448), written once (fp16 1.0 pairs)
  if (a_in_tmem && warp < 4) {
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = 0x3c003c00u;
    tc::tmem_st32u(tbase + ((uint32_t)(warp * 32) << 16) + 384, w);
    tc::tmem_st32u(tbase + ((uint32_t)(warp * 32) << 16) + 416, w);
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0) {
    const uint32_t id = tc::idesc_f16(128, N, false, false);
    const uint32_t aA = smem_u32(sA), aB = smem_u32(sB);
    const long long t0 = clock64();
    for (int i = 0; i < n_instr; ++i) {
      const int kk = ksteps == 8 ? (i & 7) : (i & 3);
      const uint32_t offA = (kk >> 2) * 16384 + (kk & 3) * 32;
      const uint32_t offB = (kk >> 2) * (N * 128) + (kk & 3) * 32;
      if (a_in_tmem)
        tc::mma_f16_ts(tbase, tbase + 384 + kk * 8, tc::smem_desc(aB + offB, 16, 1024), id, 1);
      else
        tc::mma_f16_ss(tbase, tc::smem_desc(aA + offA, 16, 1024),
                       tc::smem_desc(aB + offB, 16, 1024), id, 1);
    }
    const long long t1 = clock64();
    tc::commit(bar);
    const bool ok = mbar_wait(bar, 0);
    const long long t2 = clock64();
    if (blockIdx.x == 0) {
      cycles[0] = t1 - t0;
      cycles[1] = ok ? t2 - t0 : -1;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tbase, 512);
}

}  // namespace
}  // namespace pa

// n_instr MMAs per CTA on `grid` CTAs (one per SM); N = 128 or 256 (256 only
// with A in shared memory); ksteps = 4 or 8 (see above).  Fills cycles[0] = issue, cycles[1] = completion
// (SM clocks of CTA 0; -1 if the completion wait timed out) and *ms = the
// CUDA-event time of the timed launch (after one untimed launch).  Returns 0,
// or a negative code for invalid arguments / CUDA errors.
extern "C" __attribute__((visibility("default"))) int pa_selftest_mma_rate(
    int n_instr, int N, int a_in_tmem, int ksteps, int grid, long long* cycles, float* ms) {
  if (n_instr < 1 || grid < 1 || (N != 128 && N != 256) || (a_in_tmem && N != 128) ||
      (ksteps != 4 && ksteps != 8))
    return -1;
  if (cudaFuncSetAttribute(pa::mma_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           pa::kRateSmem) != cudaSuccess)
    return -2;
  long long* d = nullptr;
  if (cudaMalloc(&d, 2 * sizeof(long long)) != cudaSuccess) return -3;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  pa::mma_rate_kernel<<<grid, 128, pa::kRateSmem>>>(n_instr, N, a_in_tmem, ksteps, d);
  cudaEventRecord(e0);
  pa::mma_rate_kernel<<<grid, 128, pa::kRateSmem>>>(n_instr, N, a_in_tmem, ksteps, d);
  cudaEventRecord(e1);
  int rc = cudaEventSynchronize(e1) == cudaSuccess ? 0 : -4;
  if (rc == 0) {
    cudaEventElapsedTime(ms, e0, e1);
    if (cudaMemcpy(cycles, d, 2 * sizeof(long long), cudaMemcpyDeviceToHost) != cudaSuccess) rc = -5;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFree(d);
  return rc;
}
