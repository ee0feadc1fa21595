// Causal / chunked prefill over a paged KV cache on the 5th-generation tensor
// cores (sm_103a): the flash_attn_with_kvcache prefill of flash-attention #824
// "Add support for small page sizes" (reproduction: 170 new tokens, 32 heads,
// head_dim 128, 16-token pages, causal=True over a cache) and the prefill part
// of the unified varlen launch of vLLM #6052.
//
// CTA = one 128-row query tile of one query head (192 threads, 6 warps):
//   warps 0-3  softmax: thread r owns query row r = TMEM lane r.  Reads S from
//              TMEM, masks (causal, bottom-right), keeps the running max and
//              sum in the log2 domain, writes P (fp16/bf16) into shared memory
//              in the 128-byte-swizzled K-major layout, rescales O in TMEM only
//              when the running max grew by more than 2^8 (the final O / l is
//              unchanged by the choice of reference max), and does the epilogue.
//   warp 4     TMA producer: Q once, then per 128-key tile 8 pages of K and V,
//              each page resolved absolutely from the block table and fetched
//              as boxes of {64 columns, 1 head, 16 tokens}.
//   warp 5     MMA issuer + TMEM owner: S = Q K^T into one of two TMEM buffers
//              (tile j+1 is issued before P V of tile j so the tensor core runs
//              ahead of the softmax), O += P V into TMEM (V as an MN-major
//              operand).
// TMEM: S0 cols [0,128), S1 [128,256), O [256, 256+D).
#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_prefill.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // keys per tile (8 pages)
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct PrefillTraits {
  static constexpr int kHalves = D / 64;            // 64-column (128-byte) slabs
  static constexpr int kSlab = 128 * 128;           // bytes of one 128-row slab
  static constexpr int kStages = (D == 128) ? 2 : 3;
  static constexpr int kQBytes = kHalves * kSlab;
  static constexpr int kKVBytes = kHalves * kSlab;  // one K (or V) tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffP = kOffV + kStages * kKVBytes;
  static constexpr int kOffBar = kOffP + 2 * kSlab;  // P: 128 keys = 2 slabs
  static constexpr int kNumBars = 1 + 4 * kStages + 2 + 2 + 1 + 1;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
};

struct Seq {
  int qlen, lk;
  int64_t q0;  // varlen: first token row; kvcache: 0
};

__device__ __forceinline__ Seq prefill_seq(const PrefillParams& p, int b) {
  Seq s;
  int old;
  if (p.cu_seqlens_q != nullptr) {
    s.q0 = __ldg(p.cu_seqlens_q + b);
    s.qlen = __ldg(p.cu_seqlens_q + b + 1) - (int)s.q0;
    s.lk = __ldg(p.seqlens_k + b);
    old = s.lk;
  } else {
    s.q0 = 0;
    s.qlen = p.Lq;
    old = __ldg(p.cache_seqlens + b);
    s.lk = old + p.Lnew;
  }
  bool bad = old < 0 || s.lk < 0 || s.lk > p.max_seqlen_k || s.qlen < 0;
  if (p.block_table != nullptr)
    bad = bad || (int64_t)(s.lk + kPage - 1) / kPage > p.max_pages;
  else
    bad = bad || (int64_t)s.lk > p.extent;
  if (bad) {
    report(p.err, PA_DEVERR_LENGTH, b, s.lk);
    s.lk = 0;
  }
  return s;
}

template <int D, typename T>
__global__ void __launch_bounds__(192, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v) {
  using Tr = PrefillTraits<D>;
  using E = Elem<T>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + Tr::kOffQ;
  uint8_t* sK = smem + Tr::kOffK;
  uint8_t* sV = smem + Tr::kOffV;
  uint8_t* sP = smem + Tr::kOffP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* v_full = k_full + Tr::kStages;
  uint64_t* k_empty = v_full + Tr::kStages;
  uint64_t* v_empty = k_empty + Tr::kStages;
  uint64_t* s_full = v_empty + Tr::kStages;  // [2]
  uint64_t* s_free = s_full + 2;             // [2]
  uint64_t* p_full = s_free + 2;
  uint64_t* pv_done = p_full + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Tr::kOffMisc);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- which tile: heaviest (last) query tiles of every sequence first
  const int per_tile = p.B * p.Hq;
  const int tile = p.q_tiles - 1 - (int)(blockIdx.x / per_tile);
  const int rem = (int)(blockIdx.x % per_tile);
  const int b = rem / p.Hq;
  const int h = rem % p.Hq;
  const Seq sq = prefill_seq(p, b);
  if (p.cu_seqlens_q != nullptr && sq.qlen * p.G <= p.decode_rows) return;  // decode path's
  const int qs = tile * kBM;
  if (qs >= sq.qlen) return;
  const int rows_here = min(kBM, sq.qlen - qs);
  int n_keys = sq.lk;
  if (p.causal) n_keys = min(sq.lk, qs + rows_here + sq.lk - sq.qlen);
  if (n_keys < 0) n_keys = 0;
  const int n_tiles = (n_keys + kBN - 1) / kBN;
  const int g = h / p.G;

  auto out_row = [&](int qi) -> T* {
    const int64_t row = sq.q0 + (p.cu_seqlens_q ? 0 : (int64_t)b * p.Lq) + qi;
    return reinterpret_cast<T*>(p.out) + (row * p.Hq + h) * D;
  };
  auto lse_at = [&](int qi) -> float* {
    if (p.cu_seqlens_q) return p.lse + (int64_t)h * p.total_q + sq.q0 + qi;
    return p.lse + ((int64_t)b * p.Hq + h) * p.Lq + qi;
  };

  if (n_tiles == 0) {  // no visible key for any row of the tile
    if (tid < kBM && qs + tid < sq.qlen) {
      T* o = out_row(qs + tid);
      for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
      if (p.lse) *lse_at(qs + tid) = neg_inf();
    }
    return;
  }

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < Tr::kStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_free[i], 4);
    }
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    fence_mbar_init();
  }
  if (warp == 5) {
    tc::tmem_alloc(tslot, Tr::kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tS[2] = {tbase, tbase + 128};
  const uint32_t tO = tbase + 256;

  if (warp == 4) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      const uint64_t pol_kv = l2_policy_evict_last();  // K/V tiles are re-read by other q tiles
      const uint64_t pol_q = l2_policy_evict_first();
      bool failed = false;
      const int qrow = (int)(p.cu_seqlens_q ? sq.q0 + qs : qs);
      const int qb = p.cu_seqlens_q ? 0 : b;
      mbar_arrive_expect_tx(q_full, Tr::kQBytes);
      for (int hh = 0; hh < Tr::kHalves; ++hh)
        tma_load_4d(sQ + hh * Tr::kSlab, &tm_q, q_full, hh * 64, h, qrow, qb, pol_q);
      CacheGeom geom{p.block_table, p.bt_stride, p.max_pages, p.extent, 0, 0};
      const int pages_total = (n_keys + kPage - 1) / kPage;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % Tr::kStages;
        const uint32_t par = (uint32_t)((j / Tr::kStages) & 1);
        const int pg0 = j * (kBN / kPage);
        const int npg = min(kBN / kPage, pages_total - pg0);
        int c2[kBN / kPage], c3[kBN / kPage];
        for (int i = 0; i < npg; ++i) {
          const PageRef r = resolve_page(geom, b, pg0 + i);
          if (!r.ok) report(p.err, PA_DEVERR_PAGE_OOB, b, pg0 + i);
          c2[i] = r.c2;
          c3[i] = r.c3;
        }
        if (!failed && !mbar_wait(&k_empty[s], par ^ 1)) {
          report(p.err, PA_DEVERR_TIMEOUT, b, j);
          failed = true;
        }
        mbar_arrive_expect_tx(&k_full[s], (uint32_t)(npg * Tr::kHalves * 2048));
        for (int i = 0; i < npg; ++i)
          for (int hh = 0; hh < Tr::kHalves; ++hh)
            tma_load_4d(sK + s * Tr::kKVBytes + hh * Tr::kSlab + i * 2048, &tm_k, &k_full[s],
                        hh * 64, g, c2[i], c3[i], pol_kv);
        if (!failed && !mbar_wait(&v_empty[s], par ^ 1)) {
          report(p.err, PA_DEVERR_TIMEOUT, b, j);
          failed = true;
        }
        mbar_arrive_expect_tx(&v_full[s], (uint32_t)(npg * Tr::kHalves * 2048));
        for (int i = 0; i < npg; ++i)
          for (int hh = 0; hh < Tr::kHalves; ++hh)
            tma_load_4d(sV + s * Tr::kKVBytes + hh * Tr::kSlab + i * 2048, &tm_v, &v_full[s],
                        hh * 64, g, c2[i], c3[i], pol_kv);
      }
    }
  } else if (warp == 5) {
    // ======================= MMA issuer =======================
    bool failed = false;
    auto wait = [&](uint64_t* bar, uint32_t par, int where) {
      if (!failed && !mbar_wait(bar, par)) {
        report(p.err, PA_DEVERR_TIMEOUT, b, where);
        failed = true;
      }
    };
    const bool bf = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t id_qk = tc::idesc_f16(kBM, kBN, bf, false);
    const uint32_t id_pv = tc::idesc_f16(kBM, D, bf, true);
    const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP);
    auto issue_qk = [&](int j) {
      const int s = j % Tr::kStages;
      wait(&k_full[s], (uint32_t)((j / Tr::kStages) & 1), 100 + j);
      if (j >= 2) wait(&s_free[j & 1], (uint32_t)(((j - 2) >> 1) & 1), 200 + j);
      tc::fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * Tr::kSlab + (kk & 3) * 32;
          tc::mma_f16_ss(tS[j & 1], tc::smem_desc(aQ + off, 16, 1024),
                         tc::smem_desc(aK + s * Tr::kKVBytes + off, 16, 1024), id_qk, kk > 0);
        }
        tc::commit(&s_full[j & 1]);
        tc::commit(&k_empty[s]);
      }
      __syncwarp();
    };
    wait(q_full, 0, 0);
    issue_qk(0);
    for (int j = 0; j < n_tiles; ++j) {
      if (j + 1 < n_tiles) issue_qk(j + 1);
      const int s = j % Tr::kStages;
      wait(p_full, (uint32_t)(j & 1), 300 + j);
      wait(&v_full[s], (uint32_t)((j / Tr::kStages) & 1), 400 + j);
      // Keys past the tile's valid range: zero their V rows so that P = 0
      // never meets a stale or non-finite value.
      const int valid = n_keys - j * kBN;
      if (valid < kBN) {
        uint8_t* vt = sV + s * Tr::kKVBytes;
        const int nrow = kBN - valid;
        for (int idx = lane; idx < nrow * Tr::kHalves * 8; idx += 32) {
          const int r = valid + idx / (Tr::kHalves * 8);
          const int rest = idx % (Tr::kHalves * 8);
          *reinterpret_cast<uint4*>(vt + (rest >> 3) * Tr::kSlab + r * 128 + (rest & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc::fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t offp = (kk >> 2) * Tr::kSlab + (kk & 3) * 32;
          tc::mma_f16_ss(tO, tc::smem_desc(aP + offp, 16, 1024),
                         tc::smem_desc(aV + s * Tr::kKVBytes + kk * 2048, Tr::kSlab, 1024), id_pv,
                         (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc::commit(pv_done);
        tc::commit(&v_empty[s]);
      }
      __syncwarp();
    }
  } else {
    // ======================= softmax warps 0-3 =======================
    const int r = tid;  // query row within the tile == TMEM lane
    const int qi = qs + r;
    const bool row_valid = qi < sq.qlen;
    int vis_end = p.causal ? qi + sq.lk - sq.qlen + 1 : sq.lk;  // keys [0, vis_end)
    vis_end = min(vis_end, n_keys);
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    float m_use = neg_inf(), l = 0.f;
    bool failed = false;
    auto wait = [&](uint64_t* bar, uint32_t par, int where) {
      if (!failed && !mbar_wait(bar, par)) {
        report(p.err, PA_DEVERR_TIMEOUT, b, where);
        failed = true;
      }
    };
    for (int j = 0; j < n_tiles; ++j) {
      wait(&s_full[j & 1], (uint32_t)((j >> 1) & 1), 500 + j);
      tc::fence_after_sync();
      float sv[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tc::tmem_ld32(tS[j & 1] + lane_off + c * 32, sv + c * 32);
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_free[j & 1]);
      const int kv0 = j * kBN;
      float mx = neg_inf();
#pragma unroll
      for (int c = 0; c < kBN; ++c) {
        const float x = (kv0 + c < vis_end) ? sv[c] * p.scale_log2 : neg_inf();
        sv[c] = x;
        mx = fmaxf(mx, x);
      }
      const float m_new = fmaxf(m_use, mx);
      float alpha = 1.f;
      bool rescale = false;
      if (m_new != neg_inf() && (m_use == neg_inf() || m_new > m_use + kRescaleThreshold)) {
        if (m_use != neg_inf()) {
          alpha = ex2(m_use - m_new);
          rescale = true;
        }
        l *= alpha;
        m_use = m_new;
      }
      uint32_t pk[kBN / 2];
      float rs = 0.f;
      if (m_use == neg_inf()) {
#pragma unroll
        for (int c = 0; c < kBN / 2; ++c) pk[c] = 0u;
      } else {
#pragma unroll
        for (int c = 0; c < kBN / 2; ++c) {
          const float a = ex2(sv[2 * c] - m_use), bb = ex2(sv[2 * c + 1] - m_use);
          rs += a + bb;
          pk[c] = E::from_f2(a, bb);
        }
      }
      l += rs;
      if (j > 0) {
        wait(pv_done, (uint32_t)((j - 1) & 1), 600 + j);
        tc::fence_after_sync();
        if (__any_sync(0xffffffffu, rescale)) {
          const float a = rescale ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float ov[32];
            tc::tmem_ld32(tO + lane_off + c * 32, ov);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] *= a;
            tc::tmem_st32(tO + lane_off + c * 32, ov);
          }
          tc::tmem_wait_st();
        }
      }
      // P row -> swizzled K-major tile (16 chunks of 8 keys)
#pragma unroll
      for (int cc = 0; cc < kBN / 8; ++cc) {
        const int half = cc >> 3, c8 = cc & 7;
        *reinterpret_cast<uint4*>(sP + half * Tr::kSlab + r * 128 + ((c8 ^ (r & 7)) << 4)) =
            make_uint4(pk[cc * 4], pk[cc * 4 + 1], pk[cc * 4 + 2], pk[cc * 4 + 3]);
      }
      fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ---- epilogue: O / l and LSE
    wait(pv_done, (uint32_t)((n_tiles - 1) & 1), 700);
    tc::fence_after_sync();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    T* orow = row_valid ? out_row(qi) : nullptr;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float ov[32];
      tc::tmem_ld32(tO + lane_off + c * 32, ov);
      tc::tmem_wait_ld();
      if (row_valid) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          uint4 u;
          u.x = E::from_f2(ov[i] * inv, ov[i + 1] * inv);
          u.y = E::from_f2(ov[i + 2] * inv, ov[i + 3] * inv);
          u.z = E::from_f2(ov[i + 4] * inv, ov[i + 5] * inv);
          u.w = E::from_f2(ov[i + 6] * inv, ov[i + 7] * inv);
          *reinterpret_cast<uint4*>(orow + c * 32 + i) = u;
        }
      }
    }
    if (row_valid && p.lse != nullptr)
      *lse_at(qi) = l > 0.f ? (m_use + lg2(l)) * kLn2 : neg_inf();
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 5) tc::tmem_dealloc(tbase, Tr::kTmemCols);
}

template <int D, typename T>
cudaError_t launch_t(const PrefillParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t st) {
  using Tr = PrefillTraits<D>;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(
        prefill_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const long long grid = (long long)p.q_tiles * p.B * p.Hq;
  if (grid <= 0) return cudaSuccess;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_kernel<D, T><<<(unsigned)grid, 192, Tr::kSmemBytes, st>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& tm_q,
                           const CUtensorMap& tm_k, const CUtensorMap& tm_v, int D, int dtype,
                           cudaStream_t st) {
  if (D == 128 && dtype == PA_F16) return launch_t<128, __half>(p, tm_q, tm_k, tm_v, st);
  if (D == 128 && dtype == PA_BF16) return launch_t<128, __nv_bfloat16>(p, tm_q, tm_k, tm_v, st);
  if (D == 64 && dtype == PA_F16) return launch_t<64, __half>(p, tm_q, tm_k, tm_v, st);
  if (D == 64 && dtype == PA_BF16) return launch_t<64, __nv_bfloat16>(p, tm_q, tm_k, tm_v, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
