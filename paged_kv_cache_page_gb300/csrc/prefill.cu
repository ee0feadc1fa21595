// Prefill / chunked-prefill attention over a paged or contiguous KV cache on
// the 5th-generation tensor cores (sm_103a), two 128-row query tiles per CTA.
//
// The method is the tile loop of flash-attention's forward pass as the
// "Add support for small page sizes" thread describes it for a paged cache
// (per 128-row query tile: S = Q K^T over 128-key tiles, causal mask, online
// softmax, O += P V, then O / l and the LSE), with page boxes resolved
// absolutely from the block table for every tile.
//
// What is GB300-specific: a CTA holds two query tiles (2p and 2p+1 of one
// head) that share every K/V tile, each with its own softmax group, so the
// tensor core runs one tile's MMAs while the other tile's softmax runs:
//   warps 0-3  softmax of query tile 0, warps 4-7 of query tile 1; warp w
//              owns TMEM lane quarter w % 4 (tile rows 32 (w%4) .. +31), one
//              thread per row and all 128 key columns (no cross-warp max
//              exchange)
//   warp 8     TMA: both query tiles of a pair, then its K tiles
//   warp 9     TMA: V tiles
//   warp 10    TMEM owner; issues O_g += P_g V (P_g from TMEM over S_g)
//   warp 11    issues S_g = Q_g K^T (both operands in shared memory)
// TMEM: S_0, S_1, O_0, O_1 (128, 128, D, D columns).  Q K^T of a group's
// tile waits for P V of that group's previous tile (whose P occupies S_g);
// the other group's MMAs fill that gap.
//
// Work unit: the pairs i and NP-1-i of one head (NP pairs of query tiles), so
// causal units cost about the same, CTAs walking them round-robin stay in
// step, and the query tiles of a head read its K/V through L2 at about the
// same time.
#include <type_traits>

#include "pa_common.cuh"
#include "pa_engine.h"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kPM = 128;                  // rows per query tile
constexpr int kPN = 128;                  // keys per KV tile
constexpr int kPTileBoxes = kPN / kPage;  // 16-token boxes per KV tile (8)
constexpr int kPWarpK = 8, kPWarpV = 9, kPWarpPV = 10, kPWarpQK = 11;
constexpr int kPThreads = 12 * 32;
constexpr float kPRescaleThreshold = 8.0f;

template <int D>
struct PfTraits {
  static constexpr int kHalves = D / 64;         // 64-column (128-byte) slabs per row
  static constexpr int kSlab = 128 * 128;        // 128 rows x 128 bytes, 128-byte swizzle
  static constexpr int kQBytes = kHalves * kSlab;   // one query tile
  static constexpr int kKVBytes = kHalves * kSlab;  // one K or V tile
  static constexpr int kStages = (D == 128) ? 2 : 3;
  static constexpr int kOffQ = 0;                              // [2 tiles]
  static constexpr int kOffK = kOffQ + 2 * kQBytes;            // [kStages]
  static constexpr int kOffV = kOffK + kStages * kKVBytes;     // [kStages]
  static constexpr int kOffBar = kOffV + kStages * kKVBytes;
  // q_full, q_empty; k_full, v_full, k_empty, v_empty [kStages];
  // s_full, p_full, pv_done, o_free [2 groups]
  static constexpr int kNumBars = 2 + 4 * kStages + 4 * 2;
  static constexpr int kOffMisc = kOffBar + kNumBars * 8;
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + alignment slack
  static_assert(2 * 128 + 2 * D <= 512, "TMEM columns");
};

// The two query tiles of pair p of head h of sequence b.
struct Pair {
  int b, h, p;
  int lk;           // keys of the sequence
  int nrows[2];     // rows of query tile 2p + g (0: past the sequence's queries)
  int k1[2];        // keys [0, k1) visible to some row of tile g
  int nk[2];        // KV tiles of tile g
  int ntiles;       // KV tiles of the pair (max over g)
  int kend;         // keys [0, kend) read by the pair
};

__device__ __forceinline__ int pf_keys(const EngineParams& p, int b, bool rep) {
  const int old = __ldg(p.cache_seqlens + b);
  const int lk = old + p.Lnew;
  bool bad = old < 0 || lk > p.max_seqlen_k;
  if (p.block_table != nullptr)
    bad = bad || (((int64_t)(lk + kPage - 1) / kPage + (1 << p.page_shift) - 1) >> p.page_shift) >
                     p.max_pages;
  else
    bad = bad || (int64_t)lk > p.extent;
  if (bad) {
    if (rep) report(p.err, PA_DEVERR_LENGTH, b, lk);
    return 0;
  }
  return lk;
}

__device__ __forceinline__ Pair pf_pair(const EngineParams& p, int b, int h, int pr, int lk) {
  Pair q;
  q.b = b;
  q.h = h;
  q.p = pr;
  q.lk = lk;
  q.ntiles = 0;
  q.kend = 0;
#pragma unroll
  for (int g = 0; g < 2; ++g) {
    const int qs = (2 * pr + g) * kPM;
    const int nrows = max(0, min(kPM, p.Lq - qs));
    int k1 = lk;
    if (p.causal) k1 = min(lk, qs + nrows + lk - p.Lq);
    k1 = nrows > 0 ? max(0, k1) : 0;
    q.nrows[g] = nrows;
    q.k1[g] = k1;
    q.nk[g] = (k1 + kPN - 1) / kPN;
    q.ntiles = max(q.ntiles, q.nk[g]);
    q.kend = max(q.kend, k1);
  }
  return q;
}

// Unit `idx` -> its sequence, head and pairs (heavier pair first); returns the
// number of pairs (1 or 2).
__device__ __forceinline__ int pf_unit(const EngineParams& p, int idx, int np, int nu, int& b,
                                       int& h, int& pair0) {
  const int bh = idx / nu;
  const int i = idx - bh * nu;
  b = bh / p.Hq;
  h = bh - b * p.Hq;
  pair0 = np - 1 - i;
  return (np - 1 - i == i) ? 1 : 2;
}
// pair pi (0 or 1) of a unit whose first pair is pair0 (the second is
// np - 1 - pair0)
__device__ __forceinline__ int pf_pair_of(int pair0, int pi, int np) {
  return pi == 0 ? pair0 : np - 1 - pair0;
}

template <int D, typename T>
__global__ void __launch_bounds__(kPThreads, 1)
    prefill_kernel(const EngineParams p, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v) {
  using Tr = PfTraits<D>;
  using E = Elem<T>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + Tr::kOffQ;
  uint8_t* sK = smem + Tr::kOffK;
  uint8_t* sV = smem + Tr::kOffV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* v_full = k_full + Tr::kStages;
  uint64_t* k_empty = v_full + Tr::kStages;
  uint64_t* v_empty = k_empty + Tr::kStages;
  uint64_t* s_full = v_empty + Tr::kStages;  // [2]: S_g of the group's next tile computed
  uint64_t* p_full = s_full + 2;             // [2]: P_g written (and O_g rescaled)
  uint64_t* pv_done = p_full + 2;            // [2]: O_g += P_g V completed
  uint64_t* o_free = pv_done + 2;            // [2]: O_g read out by the group's epilogue
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Tr::kOffMisc);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < Tr::kStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&v_full[i], 1);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&p_full[g], 4);
      mbar_init(&pv_done[g], 1);
      mbar_init(&o_free[g], 4);
    }
    fence_mbar_init();
  }
  if (warp == kPWarpK && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == kPWarpPV) {
    tc::tmem_alloc(tslot, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  auto tS = [&](int g) { return tbase + (uint32_t)(g * 128); };
  auto tO = [&](int g) { return tbase + 256u + (uint32_t)(g * D); };

  const int qt = (p.Lq + kPM - 1) / kPM;  // query tiles per sequence
  const int np = (qt + 1) / 2;            // pairs per head
  const int nu = (np + 1) / 2;            // units per head
  const int units = p.B * p.Hq * nu;
  bool failed = false;
  auto wait = [&](uint64_t* bar, uint32_t par, int where) {
    if (!failed && !mbar_wait(bar, par)) {
      report(p.err, PA_DEVERR_TIMEOUT, -1, where);
      failed = true;
    }
  };

  if (warp == kPWarpK || warp == kPWarpV) {
    // ======================= TMA producers =======================
    // Block-table entries are read one 16-token box per lane, 32 boxes (four
    // KV tiles) at a time and a batch ahead of use; lanes 0 .. 8 * halves - 1
    // issue the boxes of a tile (box = 16 tokens x 64 columns).
    const bool is_v = warp == kPWarpV;
    const uint64_t pol_kv = l2_policy_evict_last();
    const uint64_t pol_q = l2_policy_evict_first();
    const bool paged = p.block_table != nullptr;
    uint64_t* x_full = is_v ? v_full : k_full;
    uint64_t* x_empty = is_v ? v_empty : k_empty;
    uint8_t* sX = is_v ? sV : sK;
    const CUtensorMap* tm_x = is_v ? &tm_v : &tm_k;
    int tk = 0, a = 0;
    for (int idx = blockIdx.x; idx < units; idx += gridDim.x) {
      int b, h, pair0;
      const int npair = pf_unit(p, idx, np, nu, b, h, pair0);
      const int lk = pf_keys(p, b, !is_v && lane == 0);
      const int g_kv = h / p.G;
      const int32_t* trow = paged ? p.block_table + (int64_t)b * p.bt_stride : nullptr;
      for (int pi = 0; pi < npair; ++pi) {
        const Pair pr = pf_pair(p, b, h, pf_pair_of(pair0, pi, np), lk);
        if (pr.ntiles == 0) continue;
        const int pg_end = (pr.kend + kPage - 1) / kPage;
        auto load_batch = [&](int batch) -> int {
          const int lp = 32 * batch + lane;
          const int entry = lp >> p.page_shift;
          return (paged && lp < pg_end && entry < p.max_pages) ? __ldg(trow + entry) : 0;
        };
        int cur = load_batch(0);
        int nxt = (pr.ntiles > 4) ? load_batch(1) : 0;
        for (int j = 0; j < pr.ntiles; ++j) {
          if (j > 0 && (j & 3) == 0) {
            cur = nxt;
            nxt = (j + 4 < pr.ntiles) ? load_batch((j >> 2) + 1) : 0;
          }
          const int s = tk % Tr::kStages;
          const uint32_t par = (uint32_t)((tk / Tr::kStages) & 1);
          const int pg0 = j * kPTileBoxes;
          const int npg = min(kPTileBoxes, pg_end - pg0);
          // this lane's box: page (lane % 8) of the tile, slab lane / 8
          const int my_page = lane & (kPTileBoxes - 1);
          const int my_slab = lane / kPTileBoxes;
          const int raw = __shfl_sync(0xffffffffu, cur, (j & 3) * kPTileBoxes + my_page);
          const int lp = pg0 + my_page;
          bool ok;
          int c2, c3;
          if (paged) {
            ok = (lp >> p.page_shift) < p.max_pages && raw >= 0 && (int64_t)raw < p.extent;
            c2 = ok ? (lp & ((1 << p.page_shift) - 1)) * kPage : 0;
            c3 = ok ? raw : 0;
          } else {
            ok = (int64_t)lp * kPage < p.extent;
            c2 = ok ? lp * kPage : 0;
            c3 = b;
          }
          const bool issuer = my_slab < Tr::kHalves && my_page < npg;
          if (issuer && !ok && !is_v && my_slab == 0) report(p.err, PA_DEVERR_PAGE_OOB, b, lp);
          if (lane == 0) {
            wait(&x_empty[s], par ^ 1, is_v ? 21 : 20);
            mbar_arrive_expect_tx(&x_full[s], (uint32_t)(npg * Tr::kHalves * 2048));
          }
          __syncwarp();
          if (issuer)
            tma_load_4d(sX + s * Tr::kKVBytes + my_slab * Tr::kSlab + my_page * 2048, tm_x,
                        &x_full[s], my_slab * 64, g_kv, c2, c3, pol_kv);
          __syncwarp();
          ++tk;
          if (!is_v && j == 0) {
            // both query tiles of the pair, once the previous pair's have been
            // read (after this pair's first K tile is on its way); rows past
            // the sequence's queries are filled with zeros by the copy
            if (lane == 0) {
              if (a >= 1) wait(q_empty, (uint32_t)((a - 1) & 1), 10);
              mbar_arrive_expect_tx(q_full, 2 * Tr::kQBytes);
              for (int g = 0; g < 2; ++g)
                for (int hh = 0; hh < Tr::kHalves; ++hh)
                  tma_load_4d(sQ + g * Tr::kQBytes + hh * Tr::kSlab, &tm_q, q_full, hh * 64, h,
                              (2 * pr.p + g) * kPM, b, pol_q);
            }
            __syncwarp();
          }
        }
        ++a;
      }
    }
    // every issued copy must land before the CTA leaves
    if (lane == 0) {
      for (int i = 0; i < Tr::kStages; ++i) {
        const int s = tk % Tr::kStages;
        wait(&x_empty[s], (uint32_t)(((tk / Tr::kStages) & 1) ^ 1), 30);
        ++tk;
      }
    }
    __syncwarp();
  }
  else if (warp == kPWarpQK) {
    // ======================= S = Q K^T issuer =======================
    // Per KV tile j: S_0 then S_1 (each once P V of that group's previous
    // tile, whose P occupies S_g, has completed), then the K stage is freed.
    const bool bf = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t id_qk = tc::idesc_f16(kPM, kPN, bf, false);
    const uint64_t dQ0 = tc::smem_desc(smem_u32(sQ), 16, 1024);
    const uint64_t dK0 = tc::smem_desc(smem_u32(sK), 16, 1024);
    int tk = 0, a = 0, n0 = 0, n1 = 0;
    for (int idx = blockIdx.x; idx < units; idx += gridDim.x) {
      int b, h, pair0;
      const int npair = pf_unit(p, idx, np, nu, b, h, pair0);
      const int lk = pf_keys(p, b, false);
      for (int pi = 0; pi < npair; ++pi) {
        const Pair pr = pf_pair(p, b, h, pf_pair_of(pair0, pi, np), lk);
        if (pr.ntiles == 0) continue;
        wait(q_full, (uint32_t)(a & 1), 40);
        for (int j = 0; j < pr.ntiles; ++j) {
          const int s = tk % Tr::kStages;
          wait(&k_full[s], (uint32_t)((tk / Tr::kStages) & 1), 41);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (j >= pr.nk[g]) continue;
            int& n = g ? n1 : n0;
            if (n >= 1) wait(&pv_done[g], (uint32_t)((n - 1) & 1), 42 + g);
            tc::fence_after_sync();
            if (lane == 0) {
              const uint64_t dQ = dQ0 + (uint32_t)((g * Tr::kQBytes) >> 4);
              const uint64_t dK = dK0 + (uint32_t)((s * Tr::kKVBytes) >> 4);
#pragma unroll
              for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = ((kk >> 2) * Tr::kSlab + (kk & 3) * 32) >> 4;
                tc::mma_f16_ss(tS(g), dQ + off, dK + off, id_qk, kk > 0);
              }
              tc::commit(&s_full[g]);
            }
            __syncwarp();
            ++n;
          }
          if (lane == 0) tc::commit(&k_empty[s]);
          __syncwarp();
          ++tk;
        }
        if (lane == 0) tc::commit(q_empty);  // both query tiles no longer read
        __syncwarp();
        ++a;
      }
    }
  } else if (warp == kPWarpPV) {
    // ======================= O += P V issuer =======================
    // Per KV tile j: O_0 += P_0 V, then O_1 += P_1 V (the first tile of a
    // pair once the group's previous epilogue has read O_g), then the V
    // stage is freed.
    const bool bf = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t id_pv = tc::idesc_f16(kPM, D, bf, true);
    const uint64_t dV0 = tc::smem_desc(smem_u32(sV), Tr::kSlab, 1024);
    int tk = 0, n0 = 0, n1 = 0, m0 = 0, m1 = 0;
    for (int idx = blockIdx.x; idx < units; idx += gridDim.x) {
      int b, h, pair0;
      const int npair = pf_unit(p, idx, np, nu, b, h, pair0);
      const int lk = pf_keys(p, b, false);
      for (int pi = 0; pi < npair; ++pi) {
        const Pair pr = pf_pair(p, b, h, pf_pair_of(pair0, pi, np), lk);
        if (pr.ntiles == 0) continue;
        for (int j = 0; j < pr.ntiles; ++j) {
          const int s = tk % Tr::kStages;
          wait(&v_full[s], (uint32_t)((tk / Tr::kStages) & 1), 50);
          // keys at or past the pair's end: zero their V rows, so that P = 0
          // there never meets a stale or non-finite value
          const int valid = pr.kend - j * kPN;
          if (valid < kPN) {
            uint8_t* vt = sV + s * Tr::kKVBytes;
            const int nrow = kPN - valid;
            for (int e = lane; e < nrow * Tr::kHalves * 8; e += 32) {
              const int r = valid + e / (Tr::kHalves * 8);
              const int rest = e % (Tr::kHalves * 8);
              *reinterpret_cast<uint4*>(vt + (rest >> 3) * Tr::kSlab + r * 128 + (rest & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            if (j >= pr.nk[g]) continue;
            int& n = g ? n1 : n0;
            const int m = g ? m1 : m0;
            wait(&p_full[g], (uint32_t)(n & 1), 51 + g);
            if (j == 0 && m >= 1) wait(&o_free[g], (uint32_t)((m - 1) & 1), 53 + g);
            tc::fence_after_sync();
            if (lane == 0) {
              const uint64_t dV = dV0 + (uint32_t)((s * Tr::kKVBytes) >> 4);
#pragma unroll
              for (int kk = 0; kk < kPN / 16; ++kk)
                tc::mma_f16_ts(tO(g), tS(g) + kk * 8, dV + (kk * 2048 >> 4), id_pv,
                               (j > 0 || kk > 0) ? 1u : 0u);
              tc::commit(&pv_done[g]);
            }
            __syncwarp();
            ++n;
          }
          if (lane == 0) tc::commit(&v_empty[s]);
          __syncwarp();
          ++tk;
        }
        if (pr.nk[0] > 0) ++m0;
        if (pr.nk[1] > 0) ++m1;
      }
    }
  } else if (warp < 8) {
    // ======================= softmax groups =======================
    // Thread = one row of query tile g of the pair: the row's 128 scores of a
    // KV tile from TMEM, running max (rescaling O_g only when the max grows
    // by more than 2^8), P = exp2(s - m) as 16-bit values written over the
    // tile's S_g columns, and at the end of the pair O_g / l and the LSE.
    const int g = warp >> 2, quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sc_l2 = p.scale_log2;
    int n = 0;
    for (int idx = blockIdx.x; idx < units; idx += gridDim.x) {
      int b, h, pair0;
      const int npair = pf_unit(p, idx, np, nu, b, h, pair0);
      const int lk = pf_keys(p, b, false);
      for (int pi = 0; pi < npair; ++pi) {
        const Pair pr = pf_pair(p, b, h, pf_pair_of(pair0, pi, np), lk);
        const int qi = (2 * pr.p + g) * kPM + r;
        const int nk = g ? pr.nk[1] : pr.nk[0];
        const int k1 = g ? pr.k1[1] : pr.k1[0];
        const bool valid = r < (g ? pr.nrows[1] : pr.nrows[0]);
        auto out_row = [&]() {
          return reinterpret_cast<T*>(p.out) + (((int64_t)b * p.Lq + qi) * p.Hq + h) * D;
        };
        auto lse_at = [&]() { return p.lse + ((int64_t)b * p.Hq + h) * p.Lq + qi; };
        if (nk == 0) {
          // no visible key: O = 0, LSE = -inf
          if (valid) {
            T* orow = out_row();
#pragma unroll
            for (int c = 0; c < D; c += 8)
              *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
            if (p.lse != nullptr) *lse_at() = neg_inf();
          }
          continue;
        }
        int vis_end = p.causal ? min(k1, qi + lk - p.Lq + 1) : k1;
        if (!valid) vis_end = 0;
        float m_use = neg_inf(), l = 0.f;
        for (int j = 0; j < nk; ++j) {
          wait(&s_full[g], (uint32_t)(n & 1), 60 + g);
          tc::fence_after_sync();
          float v[kPN];
#pragma unroll
          for (int c = 0; c < kPN / 32; ++c) tc::tmem_ld32(tS(g) + lane_off + c * 32, v + c * 32);
          tc::tmem_wait_ld();
          const int lim = vis_end - j * kPN;  // keys [0, lim) of the tile are visible
          const bool full = lim >= kPN;
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = neg_inf();
          if (full) {
#pragma unroll
            for (int i = 0; i < kPN; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], v[i]);
          } else {
#pragma unroll
            for (int i = 0; i < kPN; ++i) mx8[i & 7] = (i < lim) ? fmaxf(mx8[i & 7], v[i]) : mx8[i & 7];
          }
          float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                           fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
          if (mx != neg_inf()) mx *= sc_l2;
          const float m_new = fmaxf(m_use, mx);
          float alpha = 1.f;
          bool rescale = false;
          if (m_new != neg_inf() && (m_use == neg_inf() || m_new > m_use + kPRescaleThreshold)) {
            if (m_use != neg_inf()) {
              alpha = ex2(m_use - m_new);
              rescale = true;
            }
            l *= alpha;
            m_use = m_new;
          }
          // P over S_g: keys 32c .. 32c + 31 -> columns 16c .. 16c + 15
          const float neg_m = -m_use;
          float rs8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
#pragma unroll
          for (int c = 0; c < kPN / 32; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int k = c * 32 + 2 * i;
              float e0 = ex2(fmaf(v[k], sc_l2, neg_m));
              float e1 = ex2(fmaf(v[k + 1], sc_l2, neg_m));
              if (!full) {
                e0 = (k < lim) ? e0 : 0.f;
                e1 = (k + 1 < lim) ? e1 : 0.f;
              }
              rs8[i & 7] += e0 + e1;
              pk[i] = E::from_f2(e0, e1);
            }
            tc::tmem_st16u(tS(g) + lane_off + c * 16, pk);
          }
          l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
          if (j >= 1 && __any_sync(0xffffffffu, rescale)) {
            // O_g is stable once P V of the group's previous tile is done
            wait(&pv_done[g], (uint32_t)((n - 1) & 1), 62 + g);
            tc::fence_after_sync();
            const float sa = rescale ? alpha : 1.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
              float ov[32];
              tc::tmem_ld32(tO(g) + lane_off + c * 32, ov);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) ov[i] *= sa;
              tc::tmem_st32(tO(g) + lane_off + c * 32, ov);
            }
          }
          tc::tmem_wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[g]);
          ++n;
        }
        // ---- epilogue: O_g / l and the LSE, then O_g is free for the next pair
        wait(&pv_done[g], (uint32_t)((n - 1) & 1), 64 + g);
        tc::fence_after_sync();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T* orow = out_row();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float ov[32];
          tc::tmem_ld32(tO(g) + lane_off + c * 32, ov);
          tc::tmem_wait_ld();
          if (valid) {
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
        if (valid && p.lse != nullptr) *lse_at() = l > 0.f ? (m_use + lg2(l)) * kLn2 : neg_inf();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&o_free[g]);
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kPWarpPV) tc::tmem_dealloc(tbase, 512);
}

template <int D, typename T>
cudaError_t launch_t(const EngineParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, int grid, cudaStream_t st) {
  using Tr = PfTraits<D>;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(
        prefill_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  prefill_kernel<D, T><<<grid, kPThreads, Tr::kSmemBytes, st>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const EngineParams& p, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                           const CUtensorMap& tm_v, int D, int dtype, cudaStream_t st) {
  const long long qt = (p.Lq + kPM - 1) / kPM;
  const long long units = (long long)p.B * p.Hq * (((qt + 1) / 2 + 1) / 2);
  if (units <= 0) return cudaSuccess;
  const int grid = (int)(units < num_sms() ? units : num_sms());
  if (D == 128 && dtype == PA_F16) return launch_t<128, __half>(p, tm_q, tm_k, tm_v, grid, st);
  if (D == 128 && dtype == PA_BF16)
    return launch_t<128, __nv_bfloat16>(p, tm_q, tm_k, tm_v, grid, st);
  if (D == 64 && dtype == PA_F16) return launch_t<64, __half>(p, tm_q, tm_k, tm_v, grid, st);
  if (D == 64 && dtype == PA_BF16)
    return launch_t<64, __nv_bfloat16>(p, tm_q, tm_k, tm_v, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
