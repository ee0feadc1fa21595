// Encoding self-test of the tcgen05 operand layouts used by the prefill
// kernel (test infrastructure: built into libpa_selftest.so, not the product
// library).  One CTA computes, for a 128-row A:
//   C1 = A * B1^T   (A and B1 K-major, 128-byte swizzle; B1 loaded by TMA)
//   C2 = A * B2     (B2 [K=128, N=D] stored N-contiguous: MN-major operand)
//   C3 = A * B2     with A read from TMEM (written there by threads, two
//                   16-bit elements per column) -- the P tile's layout
// with A written to shared memory by threads in the swizzled K-major layout
// (the path the prefill kernel's P tile takes) and B1/B2 fetched by TMA boxes
// of 64 columns (the path of its K and V tiles).  Accumulators live in TMEM
// and are read back with tcgen05.ld by four warps.
#include <cudaTypedefs.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_tcgen05.cuh"

namespace {

using namespace pa;

template <typename T, int D>
__global__ void __launch_bounds__(192, 1)
    selftest_kernel(const T* __restrict__ A, float* __restrict__ C1, float* __restrict__ C2,
                    float* __restrict__ C3,
                    const __grid_constant__ CUtensorMap tm_b1,
                    const __grid_constant__ CUtensorMap tm_b2, int32_t* status, int a_col) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sA = smem;               // 2 halves x 128 rows x 128 B
  uint8_t* sB1 = smem + 32768;      // 2 halves x 128 rows x 128 B
  uint8_t* sB2 = smem + 65536;      // D/64 halves x 128 rows x 128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 65536 + (D / 64) * 16384);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 4);
  uint64_t* b_full = &bars[0];
  uint64_t* mma_done = &bars[1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(b_full, 1);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(tslot, 512);
    tc::tmem_relinquish();
  }
  // A rows -> swizzled K-major tile (thread t owns row t)
  if (tid < 128) {
    const T* arow = A + tid * 128;
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = *reinterpret_cast<const uint4*>(arow + c * 8);
      const int half = c >> 3, cc = c & 7;
      *reinterpret_cast<uint4*>(sA + half * 16384 + tid * 128 + ((cc ^ (tid & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  // A rows -> TMEM columns [384, 448): thread r (warps 0-3) owns lane r
  if (tid < 128) {
    const T* arow = A + tid * 128;
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16) + 384;
    for (int c = 0; c < 2; ++c) {
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = *reinterpret_cast<const uint32_t*>(arow + c * 64 + 2 * i);
      tc::tmem_st32u(lane_addr + c * 32, w);
      tc::tmem_st32u(lane_addr + 64 + c * 32, w);  // second copy at column 448
    }
    tc::tmem_wait_st();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  if (warp == 4 && lane == 0) {
    mbar_arrive_expect_tx(b_full, 32768 + (D / 64) * 16384);
    for (int h = 0; h < 2; ++h)
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(sB1 + h * 16384)),
          "l"(reinterpret_cast<uint64_t>(&tm_b1)), "r"(h * 64), "r"(0), "r"(smem_u32(b_full))
          : "memory");
    for (int h = 0; h < D / 64; ++h)
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(sB2 + h * 16384)),
          "l"(reinterpret_cast<uint64_t>(&tm_b2)), "r"(h * 64), "r"(0), "r"(smem_u32(b_full))
          : "memory");
  }
  if (warp == 5 && lane == 0) {
    bool ok = mbar_wait(b_full, 0);
    if (!ok) atomicExch(status, 1);
    tc::fence_after_sync();
    const uint32_t id1 = tc::idesc_f16(128, 128, std::is_same<T, __nv_bfloat16>::value, false);
    const uint32_t id2 = tc::idesc_f16(128, D, std::is_same<T, __nv_bfloat16>::value, true);
    const uint32_t aA = smem_u32(sA), aB1 = smem_u32(sB1), aB2 = smem_u32(sB2);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      tc::mma_f16_ss(tbase, tc::smem_desc(aA + off, 16, 1024), tc::smem_desc(aB1 + off, 16, 1024),
                     id1, kk > 0);
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t offA = (kk >> 2) * 16384 + (kk & 3) * 32;
      tc::mma_f16_ss(tbase + 128, tc::smem_desc(aA + offA, 16, 1024),
                     tc::smem_desc(aB2 + kk * 2048, 16384, 1024), id2, kk > 0);
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
      tc::mma_f16_ts(tbase + 256, tbase + a_col + kk * 8,
                     tc::smem_desc(aB2 + kk * 2048, 16384, 1024), id2, kk > 0);
    tc::commit(mma_done);
  }
  if (warp < 4) {
    if (!mbar_wait(mma_done, 0)) atomicExch(status, 2);
    tc::fence_after_sync();
    const int row = warp * 32 + lane;
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    float v[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      tc::tmem_ld32(lane_addr + c * 32, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) C1[row * 128 + c * 32 + i] = v[i];
    }
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      tc::tmem_ld32(lane_addr + 128 + c * 32, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) C2[row * D + c * 32 + i] = v[i];
    }
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      tc::tmem_ld32(lane_addr + 256 + c * 32, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) C3[row * D + c * 32 + i] = v[i];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 5) tc::tmem_dealloc(tbase, 512);
}

bool encode2d(CUtensorMap* m, const void* base, int dtype, uint64_t cols, uint64_t rows) {
  void* fnp = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return false;
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fnp);
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
            2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, int D>
int run(const void* A, const void* B1, const void* B2, float* C1, float* C2, float* C3,
        int32_t* status, int a_col, cudaStream_t st) {
  CUtensorMap m1, m2;
  if (!encode2d(&m1, B1, std::is_same<T, __nv_bfloat16>::value ? PA_BF16 : PA_F16, 128, 128) ||
      !encode2d(&m2, B2, std::is_same<T, __nv_bfloat16>::value ? PA_BF16 : PA_F16, D, 128))
    return -1;
  const int smem = 1024 + 65536 + (D / 64) * 16384 + 256;
  if (cudaFuncSetAttribute(selftest_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -2;
  selftest_kernel<T, D><<<1, 192, smem, st>>>(reinterpret_cast<const T*>(A), C1, C2, C3, m1,
                                              m2, status, a_col);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int pa_selftest_tcgen05_gemm(
    const void* A, const void* B1, const void* B2, float* C1, float* C2, float* C3, int D,
    int dtype, int32_t* status, int a_col, cudaStream_t st) {
  if (a_col != 384 && a_col != 448) return -5;
  if (D == 128 && dtype == PA_F16) return run<__half, 128>(A, B1, B2, C1, C2, C3, status, a_col, st);
  if (D == 128 && dtype == PA_BF16)
    return run<__nv_bfloat16, 128>(A, B1, B2, C1, C2, C3, status, a_col, st);
  if (D == 64 && dtype == PA_F16) return run<__half, 64>(A, B1, B2, C1, C2, C3, status, a_col, st);
  if (D == 64 && dtype == PA_BF16)
    return run<__nv_bfloat16, 64>(A, B1, B2, C1, C2, C3, status, a_col, st);
  return -4;
}
