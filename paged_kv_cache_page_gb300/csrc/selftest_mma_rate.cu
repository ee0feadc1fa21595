// Tensor-core rate of the attention MMA shapes (test-only library): every CTA
// (one per SM) issues `n_instr` back-to-back kind::f16 MMAs of M = 128,
// K = 16 and N in {128, 256} into one TMEM accumulator, A from shared memory
// or from TMEM, and its first thread times issue and completion with the SM
// clock.  Every group of 8 instructions walks the 8 k-steps of a K = 128
// product over two 128-byte-swizzled slabs, so each instruction reads distinct
// operand bytes, as the attention tiles do.
//   lean = 1: descriptors built once, k-steps unrolled with constant offsets
//             (the issuing thread spends a few instructions per MMA);
//   lean = 0: descriptors rebuilt per instruction in a runtime loop.
// The two show how much of an MMA stream's rate the single issuing thread's
// own instructions can cost: at N = 128 the tensor pipe takes about 64 SM
// cycles per instruction, close to what a thread spends building two
// descriptors and the loop around them.
#include <cuda_runtime.h>

#include "pa_common.cuh"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kRateSmem = 120 * 1024;  // one CTA per SM

template <int N, bool kTS, bool kLean>
__global__ void __launch_bounds__(128, 1) mma_rate_kernel(int n_instr, long long* cycles) {
  constexpr bool a_in_tmem = kTS;
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
    if (kLean) {
      const uint64_t dA = tc::smem_desc(aA, 16, 1024);
      const uint64_t dB = tc::smem_desc(aB, 16, 1024);
      constexpr uint32_t slabB = (uint32_t)(N * 128) >> 4;  // second slab of B, descriptor units
      for (int o = 0; o < n_instr / 8; ++o) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t offA = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          const uint32_t offB = (kk >> 2) * slabB + (((kk & 3) * 32) >> 4);
          if (a_in_tmem)
            tc::mma_f16_ts(tbase, tbase + 384 + kk * 8, dB + offB, id, 1);
          else
            tc::mma_f16_ss(tbase, dA + offA, dB + offB, id, 1);
        }
      }
    } else {
      for (int i = 0; i < n_instr / 8 * 8; ++i) {
        const int kk = i & 7;
        const uint32_t offA = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t offB = (kk >> 2) * (N * 128) + (kk & 3) * 32;
        if (a_in_tmem)
          tc::mma_f16_ts(tbase, tbase + 384 + kk * 8, tc::smem_desc(aB + offB, 16, 1024), id, 1);
        else
          tc::mma_f16_ss(tbase, tc::smem_desc(aA + offA, 16, 1024),
                         tc::smem_desc(aB + offB, 16, 1024), id, 1);
      }
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

template <int N, bool kTS, bool kLean>
int run(int n_instr, int grid, long long* d, float* ms) {
  if (cudaFuncSetAttribute(mma_rate_kernel<N, kTS, kLean>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, kRateSmem) != cudaSuccess)
    return -2;
  cudaEvent_t e0, e1;
  cudaEventCreate(&e0);
  cudaEventCreate(&e1);
  mma_rate_kernel<N, kTS, kLean><<<grid, 128, kRateSmem>>>(n_instr, d);
  cudaEventRecord(e0);
  mma_rate_kernel<N, kTS, kLean><<<grid, 128, kRateSmem>>>(n_instr, d);
  cudaEventRecord(e1);
  int rc = cudaEventSynchronize(e1) == cudaSuccess ? 0 : -4;
  if (rc == 0) cudaEventElapsedTime(ms, e0, e1);
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  return rc;
}

}  // namespace
}  // namespace pa

// n_instr (a multiple of 8) MMAs per CTA on `grid` CTAs (one per SM); N = 128
// or 256 (256 only with A in shared memory); lean = 1 or 0 (see above).
// Fills cycles[0] = issue, cycles[1] = completion (SM clocks of CTA 0; -1 if
// the completion wait timed out) and *ms = the CUDA-event time of the timed
// launch (after one untimed launch).  Returns 0, or a negative code for
// invalid arguments / CUDA errors.
extern "C" __attribute__((visibility("default"))) int pa_selftest_mma_rate(
    int n_instr, int N, int a_in_tmem, int lean, int grid, long long* cycles, float* ms) {
  if (n_instr < 8 || n_instr % 8 != 0 || grid < 1 || (N != 128 && N != 256) ||
      (a_in_tmem && N != 128) || (lean != 0 && lean != 1))
    return -1;
  long long* d = nullptr;
  if (cudaMalloc(&d, 2 * sizeof(long long)) != cudaSuccess) return -3;
  int rc;
  if (N == 256)
    rc = lean ? pa::run<256, false, true>(n_instr, grid, d, ms)
              : pa::run<256, false, false>(n_instr, grid, d, ms);
  else if (a_in_tmem)
    rc = lean ? pa::run<128, true, true>(n_instr, grid, d, ms)
              : pa::run<128, true, false>(n_instr, grid, d, ms);
  else
    rc = lean ? pa::run<128, false, true>(n_instr, grid, d, ms)
              : pa::run<128, false, false>(n_instr, grid, d, ms);
  if (rc == 0 && cudaMemcpy(cycles, d, 2 * sizeof(long long), cudaMemcpyDeviceToHost) != cudaSuccess)
    rc = -5;
  cudaFree(d);
  return rc;
}
