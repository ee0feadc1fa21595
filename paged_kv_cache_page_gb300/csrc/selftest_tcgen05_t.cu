// Encoding self-test of the transposed decode-tile MMA shapes (test
// infrastructure: built into libpa_selftest.so, not the product library).
// One CTA, head dim 128:
//   C4 = K Q^T    M = 128 keys, N = 16 query rows, K = 128: A = a 128-key K
//                 tile and B = the first 16 rows of a 128-row Q tile, both
//                 fetched by TMA boxes of 64 columns (K-major, 128-byte swizzle)
//   C5 = V^T P^T  M = 128 (head dim), N = 16, K = 128 keys: A = a 128-key V tile
//                 (TMA, the same layout) read as an MN-major operand, B = a
//                 16-row x 128-key P tile written by threads (K-major, 128-byte
//                 swizzle, 2 KB per 64-key slab)
// Accumulators (M rows on TMEM lanes, 16 columns) are read back by four warps.
#include <cudaTypedefs.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_tcgen05.cuh"

namespace {

using namespace pa;

template <typename T>
__global__ void __launch_bounds__(192, 1)
    selftest_t_kernel(const T* __restrict__ P, float* __restrict__ C4, float* __restrict__ C5,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_v, int32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sK = smem;            // 2 slabs x 128 rows x 128 B
  uint8_t* sQ = smem + 32768;    // 2 slabs x 128 rows x 128 B
  uint8_t* sV = smem + 65536;    // 2 slabs x 128 rows x 128 B
  uint8_t* sP = smem + 98304;    // 2 slabs x 16 rows x 128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 98304 + 4096);
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
  // P (16 x 128, row-major) -> K-major tile: element (r, key) in slab key / 64,
  // row r, 16-byte chunk ((key % 64) / 8) ^ (r % 8)
  if (tid < 128) {
    for (int e = tid; e < 16 * 128; e += 128) {
      const int r = e / 128, key = e % 128;
      const int kc = key % 64;
      T* dst = reinterpret_cast<T*>(sP + (key / 64) * 2048 + r * 128 +
                                    (((kc / 8) ^ (r & 7)) << 4)) +
               (kc % 8);
      *dst = P[e];
    }
    fence_proxy_async_smem();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;

  if (warp == 4 && lane == 0) {
    mbar_arrive_expect_tx(b_full, 3 * 32768);
    for (int h = 0; h < 2; ++h) {
      uint8_t* dsts[3] = {sK + h * 16384, sQ + h * 16384, sV + h * 16384};
      const CUtensorMap* maps[3] = {&tm_k, &tm_q, &tm_v};
      for (int m = 0; m < 3; ++m)
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dsts[m])),
            "l"(reinterpret_cast<uint64_t>(maps[m])), "r"(h * 64), "r"(0), "r"(smem_u32(b_full))
            : "memory");
    }
  }
  if (warp == 5 && lane == 0) {
    bool ok = mbar_wait(b_full, 0);
    if (!ok) atomicExch(status, 1);
    tc::fence_after_sync();
    const bool bf = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t id4 = tc::idesc_f16_mn(128, 16, bf, false, false);
    const uint32_t id5 = tc::idesc_f16_mn(128, 16, bf, true, false);
    const uint32_t aK = smem_u32(sK), aQ = smem_u32(sQ), aV = smem_u32(sV), aP = smem_u32(sP);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
      tc::mma_f16_ss(tbase, tc::smem_desc(aK + off, 16, 1024), tc::smem_desc(aQ + off, 16, 1024),
                     id4, kk > 0);
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t offp = (kk >> 2) * 2048 + (kk & 3) * 32;
      tc::mma_f16_ss(tbase + 128, tc::smem_desc(aV + kk * 2048, 16384, 1024),
                     tc::smem_desc(aP + offp, 16, 1024), id5, kk > 0);
    }
    tc::commit(mma_done);
  }
  if (warp < 4) {
    if (!mbar_wait(mma_done, 0)) atomicExch(status, 2);
    tc::fence_after_sync();
    const int row = warp * 32 + lane;
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    float v[16];
    tc::tmem_ld16(lane_addr, v);
    tc::tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) C4[row * 16 + i] = v[i];
    tc::tmem_ld16(lane_addr + 128, v);
    tc::tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) C5[row * 16 + i] = v[i];
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 5) tc::tmem_dealloc(tbase, 512);
}

bool encode2d(CUtensorMap* m, const void* base, int dtype) {
  void* fnp = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return false;
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fnp);
  const cuuint64_t dims[2] = {128, 128};
  const cuuint64_t strides[1] = {128 * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
            2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
int run(const void* K, const void* Q, const void* V, const void* P, float* C4, float* C5,
        int32_t* status, cudaStream_t st) {
  const int dt = std::is_same<T, __nv_bfloat16>::value ? PA_BF16 : PA_F16;
  CUtensorMap mk, mq, mv;
  if (!encode2d(&mk, K, dt) || !encode2d(&mq, Q, dt) || !encode2d(&mv, V, dt)) return -1;
  const int smem = 1024 + 98304 + 4096 + 256;
  if (cudaFuncSetAttribute(selftest_t_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -2;
  selftest_t_kernel<T><<<1, 192, smem, st>>>(reinterpret_cast<const T*>(P), C4, C5, mk, mq, mv,
                                             status);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace

// K, Q, V: 128 x 128 row-major; P: 16 x 128 row-major; C4, C5: 128 x 16 fp32.
extern "C" __attribute__((visibility("default"))) int pa_selftest_tcgen05_transposed(
    const void* K, const void* Q, const void* V, const void* P, float* C4, float* C5, int dtype,
    int32_t* status, cudaStream_t st) {
  if (dtype == PA_F16) return run<__half>(K, Q, V, P, C4, C5, status, st);
  if (dtype == PA_BF16) return run<__nv_bfloat16>(K, Q, V, P, C4, C5, status, st);
  return -4;
}

// ---------------------------------------------------------------------------
// Q copied into TMEM by tcgen05.cp: C1 = Q K^T with Q from shared memory and
// C2 = Q K^T with Q from TMEM (after eight 128x256b copies of the 128-byte-
// swizzled Q tile, one per 16-element k-step), M = N = K = 128.
namespace {

template <typename T>
__global__ void __launch_bounds__(192, 1)
    selftest_cpq_kernel(float* __restrict__ C1, float* __restrict__ C2,
                        const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k, int32_t* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem;            // 2 slabs x 128 rows x 128 B
  uint8_t* sK = smem + 32768;    // 2 slabs x 128 rows x 128 B
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 65536);
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
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  if (warp == 4 && lane == 0) {
    mbar_arrive_expect_tx(b_full, 2 * 32768);
    for (int h = 0; h < 2; ++h) {
      uint8_t* dsts[2] = {sQ + h * 16384, sK + h * 16384};
      const CUtensorMap* maps[2] = {&tm_q, &tm_k};
      for (int m = 0; m < 2; ++m)
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dsts[m])),
            "l"(reinterpret_cast<uint64_t>(maps[m])), "r"(h * 64), "r"(0), "r"(smem_u32(b_full))
            : "memory");
    }
  }
  if (warp == 5 && lane == 0) {
    if (!mbar_wait(b_full, 0)) atomicExch(status, 1);
    tc::fence_after_sync();
    const bool bf = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t id = tc::idesc_f16(128, 128, bf, false);
    const uint64_t dQ = tc::smem_desc(smem_u32(sQ), 16, 1024);
    const uint64_t dK = tc::smem_desc(smem_u32(sK), 16, 1024);
    const uint32_t tQ = tbase + 256;  // Q in TMEM: 64 columns (two 16-bit values each)
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
      tc::cp_128x256b(tQ + kk * 8, dQ + off);
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
      tc::mma_f16_ss(tbase, dQ + off, dK + off, id, kk > 0);
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint32_t off = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
      tc::mma_f16_ts(tbase + 128, tQ + kk * 8, dK + off, id, kk > 0);
    }
    tc::commit(mma_done);
  }
  if (warp < 4) {
    if (!mbar_wait(mma_done, 0)) atomicExch(status, 2);
    tc::fence_after_sync();
    const int row = warp * 32 + lane;
    const uint32_t lane_addr = tbase + ((uint32_t)(warp * 32) << 16);
    for (int c = 0; c < 128; c += 32) {
      float v[32];
      tc::tmem_ld32(lane_addr + c, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) C1[row * 128 + c + i] = v[i];
      tc::tmem_ld32(lane_addr + 128 + c, v);
      tc::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) C2[row * 128 + c + i] = v[i];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 5) tc::tmem_dealloc(tbase, 512);
}

template <typename T>
int run_cpq(const void* Q, const void* K, float* C1, float* C2, int32_t* status, cudaStream_t st) {
  const int dt = std::is_same<T, __nv_bfloat16>::value ? PA_BF16 : PA_F16;
  CUtensorMap mq, mk;
  if (!encode2d(&mq, Q, dt) || !encode2d(&mk, K, dt)) return -1;
  const int smem = 1024 + 65536 + 256;
  if (cudaFuncSetAttribute(selftest_cpq_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem) != cudaSuccess)
    return -2;
  selftest_cpq_kernel<T><<<1, 192, smem, st>>>(C1, C2, mq, mk, status);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // namespace

// Q, K: 128 x 128 row-major; C1, C2: 128 x 128 fp32 (Q K^T, Q from shared
// memory and from TMEM after tcgen05.cp).
extern "C" __attribute__((visibility("default"))) int pa_selftest_tcgen05_cpq(
    const void* Q, const void* K, float* C1, float* C2, int dtype, int32_t* status,
    cudaStream_t st) {
  if (dtype == PA_F16) return run_cpq<__half>(Q, K, C1, C2, status, st);
  if (dtype == PA_BF16) return run_cpq<__nv_bfloat16>(Q, K, C1, C2, status, st);
  return -4;
}
