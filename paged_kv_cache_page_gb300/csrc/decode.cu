// Split-KV paged decode for GB300 (sm_103a).
//
// One work item = (sequence b, kv head g, split s): the Lq_b * G query rows
// that share kv head g (GQA-packed, so K/V are streamed once per kv head)
// against the keys of split s.  A persistent grid of CTAs walks the item list
// that every CTA derives on the GPU from the sequence lengths (the device-side
// replacement of a host num_splits heuristic, which would need the lengths on
// the CPU: flash-attention #1000 "Inappropriate Number of Splits ...").
//
// CTA = 1 producer warp + 8 consumer warps.  The producer resolves every
// 16-token page absolutely from the block table (flash-attention #824 "Add
// support for small page sizes": one page per fetch, each from its own table
// entry; the relative page-delta bug discussed there cannot arise), reading
// the entries warp-wide 32 at a time one batch ahead of use, and issues one
// TMA box {D, 1 head, 16 tokens} per page for K and for V from eight lanes into
// a shared-memory ring of 4-page stages.  Consumer warps w and w + 4 own page w
// of a stage, 8 keys each (two warps per page double the warps that hide the
// latency of the per-key dependency chains): QK^T with 8 lanes per key
// (16-byte shared loads), fp32 online softmax in the log2 domain, PV with each
// lane owning D/32 output columns.  The eight warps' (m, l, O) are merged at
// the end of the item and written either as the final output (one split) or
// as a normalised partial + LSE for the combine step.
//
// New tokens of a kvcache call (k=/v= append) are patched into the staged page
// from k_new/v_new and written to their cache slots by the CTA whose split
// covers them, so no CTA ever reads a slot another CTA is writing.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

template <int D, typename T, int RMAX>
struct DecodeTraits {
  static constexpr int kStagePages = 4;
  static constexpr int kKeyParts = 2;  // consumer warps per page, 16 / kKeyParts keys each
  static constexpr int kPartKeys = kPage / kKeyParts;
  static constexpr int kConsumerWarps = kStagePages * kKeyParts;
  static constexpr int kThreads = (kConsumerWarps + 1) * 32;
  static constexpr int kStages = (D == 128) ? 3 : 5;
  static constexpr int kPageElems = kPage * D;
  static constexpr int kPageBytes = kPageElems * 2;
  static constexpr int kQCh = D / 64;  // 16-byte chunks per lane per key in QK
  static constexpr int kPVE = D / 32;  // output columns per lane
  // shared memory layout (bytes)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kStagePages * kPageBytes;
  static constexpr int kOffMerge = kOffV + kStages * kStagePages * kPageBytes;
  static constexpr int kMergeFloats = (kConsumerWarps - 1) * RMAX * (D + 2);
  static constexpr int al16(int x) { return (x + 15) & ~15; }
  static constexpr int kOffPrefix = al16(kOffMerge + kMergeFloats * 4);
  static constexpr int kOffInfo = al16(kOffPrefix + (kDecodeMaxSchedB + 1) * 4);
  static constexpr int kOffBar = al16(kOffInfo + kStages * kStagePages * 12);
  static constexpr int kOffMisc = al16(kOffBar + 2 * kStages * 8);
  static constexpr int kOffQ = kOffMisc + 64;  // [stage][RMAX][D] query rows of an item
  static constexpr int kQRowBytes = D * 2;
  static constexpr int kSmemBytes = ((kOffQ + kStages * RMAX * kQRowBytes) + 127) & ~127;
  static_assert(kOffBar % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(kOffV % 128 == 0, "TMA destinations need 128-byte alignment");
};

struct SeqInfo {
  int qlen;     // query rows of this sequence
  int64_t row0;  // global row index of its first query row (NR addressing)
  int lk;       // keys attended
  int old;      // keys already in the cache (kvcache); == lk in varlen mode
  bool active;  // has decode work (varlen: rows * G <= RMAX)
};

template <int RMAX>
__device__ __forceinline__ SeqInfo seq_info(const DecodeParams& p, int b, bool report_errors) {
  SeqInfo si;
  if (p.cu_seqlens_q != nullptr) {
    const int q0 = __ldg(p.cu_seqlens_q + b), q1 = __ldg(p.cu_seqlens_q + b + 1);
    si.qlen = q1 - q0;
    si.row0 = q0;
    si.lk = __ldg(p.seqlens_k + b);
    si.old = si.lk;
    si.active = si.qlen > 0 && si.qlen * p.G <= RMAX;
  } else {
    si.qlen = p.Lq;
    si.row0 = (int64_t)b * p.Lq;
    si.old = __ldg(p.cache_seqlens + b);
    si.lk = si.old + p.Lnew;
    si.active = true;
  }
  bool bad = si.old < 0 || si.lk < 0 || si.lk > p.max_seqlen_k || si.qlen < 0;
  if (p.block_table != nullptr) {
    bad = bad || (((int64_t)(si.lk + kPage - 1) / kPage + (1 << p.page_shift) - 1) >> p.page_shift) >
                     p.max_pages;
  } else {
    bad = bad || (int64_t)si.lk > p.extent;
  }
  if (bad) {
    if (report_errors) report(p.err, PA_DEVERR_LENGTH, b, si.lk);
    si.lk = 0;
    si.old = 0;
  }
  return si;
}

template <int D, typename T, int RMAX>
__global__ void __launch_bounds__(DecodeTraits<D, T, RMAX>::kThreads, 2)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  using Tr = DecodeTraits<D, T, RMAX>;
  using E = Elem<T>;
  extern __shared__ __align__(1024) uint8_t smem[];
  T* sK = reinterpret_cast<T*>(smem + Tr::kOffK);
  T* sV = reinterpret_cast<T*>(smem + Tr::kOffV);
  float* sMerge = reinterpret_cast<float*>(smem + Tr::kOffMerge);
  int* sPrefix = reinterpret_cast<int*>(smem + Tr::kOffPrefix);
  int* sInfo = reinterpret_cast<int*>(smem + Tr::kOffInfo);  // [stage][page][c2, c3, ok]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Tr::kOffBar);
  uint64_t* empty = full + Tr::kStages;
  int* sMisc = reinterpret_cast<int*>(smem + Tr::kOffMisc);
  T* sQ = reinterpret_cast<T*>(smem + Tr::kOffQ);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < Tr::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], Tr::kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == Tr::kConsumerWarps && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }

  // ---- device split schedule: per-sequence split counts and their prefix sum
  const bool direct = p.s_max <= 1 && p.cu_seqlens_q == nullptr;
  int num_items;
  int chunk = 0;
  if (direct) {
    num_items = p.B * p.Hkv;
  } else {
    // pages of every sequence -> sPrefix (scratch until the prefix sum
    // replaces it) and the longest one (block max); then the cost of each
    // candidate split count (block sums of the work items it makes)
    SplitSched sch{p.s_max, p.target_ctas, p.min_chunk_pages};
    int* sRed = reinterpret_cast<int*>(sMerge);  // [warp][kSplitCands]
    int pmax = 0;
    for (int b = tid; b < p.B; b += Tr::kThreads) {
      SeqInfo si = seq_info<RMAX>(p, b, true);
      const int pages = si.active ? (si.lk + kPage - 1) / kPage : -1;
      sPrefix[b] = pages;
      pmax = max(pmax, pages);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
    if (lane == 0) sRed[warp] = pmax;
    __syncthreads();
    pmax = 0;
    for (int w = 0; w < Tr::kThreads / 32; ++w) pmax = max(pmax, sRed[w]);
    __syncthreads();
    if (p.target_ctas >= kForcedSplitTarget) {
      chunk = max(1, p.min_chunk_pages);
    } else {
      int cchunk[kSplitCands], cnt[kSplitCands];
#pragma unroll
      for (int i = 0; i < kSplitCands; ++i) {
        cchunk[i] = split_cand_chunk(sch, pmax, split_cand(i));
        cnt[i] = 0;
      }
      for (int b = tid; b < p.B; b += Tr::kThreads) {
        const int pages = sPrefix[b];
        if (pages < 0) continue;
#pragma unroll
        for (int i = 0; i < kSplitCands; ++i) {
          int n;
          split_pages_per(sch, pages, cchunk[i], &n);
          cnt[i] += n;
        }
      }
#pragma unroll
      for (int i = 0; i < kSplitCands; ++i) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cnt[i] += __shfl_xor_sync(0xffffffffu, cnt[i], o);
      }
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kSplitCands; ++i) sRed[warp * kSplitCands + i] = cnt[i];
      }
      __syncthreads();
      int best = -1;
#pragma unroll
      for (int i = 0; i < kSplitCands; ++i) {
        const int n = split_cand(i);
        if (n <= max(1, p.s_max)) {
          int items = 0;
          for (int w = 0; w < Tr::kThreads / 32; ++w) items += sRed[w * kSplitCands + i];
          const int cost = split_cand_cost(sch, items * p.Hkv, cchunk[i], n > 1);
          if (best < 0 || cost < best) {
            best = cost;
            chunk = cchunk[i];
          }
        }
      }
      __syncthreads();
    }
    if (warp == 0) {
      int carry = 0;
      for (int base = 0; base < p.B; base += 32) {
        const int b = base + lane;
        int n = 0;
        if (b < p.B) {
          const int pages = sPrefix[b];
          if (pages >= 0) split_pages_per(sch, pages, chunk, &n);
          // split count read by the combine step, for every sequence (0: the
          // sequence's rows are written directly)
          if (blockIdx.x == 0 && p.nsplit != nullptr) p.nsplit[b] = n > 1 ? n : 0;
        }
        int incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (b < p.B) sPrefix[b] = carry + incl - n;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        sPrefix[p.B] = carry;
        sMisc[0] = carry;
      }
    }
    __syncthreads();
    num_items = sMisc[0] * p.Hkv;
  }
  __syncthreads();

  const SplitSched sch{p.s_max, p.target_ctas, p.min_chunk_pages};

  // Work-item decoding shared by producer and consumers.
  auto item_of = [&](int item, int& b, int& g, int& s, int& nb, int& p0, int& p1, SeqInfo& si) {
    g = item % p.Hkv;
    const int j = item / p.Hkv;
    if (direct) {
      b = j;
      s = 0;
    } else {
      int lo = 0, hi = p.B;  // find last b with prefix[b] <= j
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sPrefix[mid] <= j) lo = mid; else hi = mid;
      }
      b = lo;
      s = j - sPrefix[b];
    }
    si = seq_info<RMAX>(p, b, true);
    const int pages = (si.lk + kPage - 1) / kPage;
    const int per = direct ? pages : split_pages_per(sch, pages, chunk, &nb);
    if (direct) nb = 1;
    p0 = s * per;
    p1 = min(p0 + per, pages);
    if (p0 > p1) p0 = p1;
  };

  // the combine grid that follows may be scheduled now; it waits on the
  // device for this grid's completion before reading any partial
  griddep_launch_dependents();
  const int cta = blockIdx.x;
  const int num_ctas = gridDim.x;

  if (warp == Tr::kConsumerWarps) {
    // ======================= producer warp =======================
    // The block-table entries of the item are read warp-wide, one page per
    // lane, 32 pages at a time and one batch ahead, so no stage waits on a
    // table load.  Lanes 0-3 issue the K boxes and lanes 4-7 the V boxes of
    // a stage's pages.
    const uint64_t pol = l2_policy_evict_first();
    CacheGeom geom{p.block_table, p.bt_stride, p.max_pages, p.extent, p.k_sb, p.k_st, p.page_shift};
    int stage = 0;
    uint32_t phase = 0;
    bool failed = false;
    auto fetch = [&](int b, int lp, int p1, int& c2, int& c3, int& ok) {
      c2 = 0;
      c3 = 0;
      ok = 0;
      if (lp < p1) {
        const PageRef r = resolve_page(geom, b, lp);
        if (!r.ok) report(p.err, PA_DEVERR_PAGE_OOB, b, lp);
        c2 = r.c2;
        c3 = r.c3;
        ok = r.ok ? 1 : 0;
      }
    };
    for (int item = cta; item < num_items; item += num_ctas) {
      int b, g, s, nb, p0, p1;
      SeqInfo si;
      item_of(item, b, g, s, nb, p0, p1, si);
      int base = p0;
      int cur2, cur3, curok, nxt2, nxt3, nxtok;
      fetch(b, p0 + lane, p1, cur2, cur3, curok);
      fetch(b, p0 + 32 + lane, p1, nxt2, nxt3, nxtok);
      for (int pg = p0; pg < p1; pg += Tr::kStagePages) {
        if (pg - base >= 32) {
          base += 32;
          cur2 = nxt2;
          cur3 = nxt3;
          curok = nxtok;
          fetch(b, base + 32 + lane, p1, nxt2, nxt3, nxtok);
        }
        if (lane == 0 && !failed && !mbar_wait(&empty[stage], phase ^ 1)) {
          report(p.err, PA_DEVERR_TIMEOUT, b, pg);
          failed = true;
        }
        __syncwarp();
        const int n = min(Tr::kStagePages, p1 - pg);
        const int w = lane & (Tr::kStagePages - 1);
        const int src = pg - base + w;
        const int c2 = __shfl_sync(0xffffffffu, cur2, src);
        const int c3 = __shfl_sync(0xffffffffu, cur3, src);
        const int ok = __shfl_sync(0xffffffffu, curok, src);
        if (lane < Tr::kStagePages && w < n) {
          int* info = sInfo + (stage * Tr::kStagePages + w) * 3;
          info[0] = c2;
          info[1] = c3;
          info[2] = ok;
        }
        __syncwarp();
        // the item's query rows travel with its first stage
        const int nq = (pg == p0) ? si.qlen * p.G : 0;
        if (lane == 0)
          mbar_arrive_expect_tx(&full[stage],
                                (uint32_t)(n * 2 * Tr::kPageBytes + nq * Tr::kQRowBytes));
        __syncwarp();
        if (lane < nq) {
          const int qi = lane / p.G;
          const int h = g * p.G + (lane % p.G);
          const T* qrow =
              p.cu_seqlens_q != nullptr
                  ? reinterpret_cast<const T*>(p.q) + (si.row0 + qi) * p.q_st + (int64_t)h * p.q_sh
                  : reinterpret_cast<const T*>(p.q) + (int64_t)b * p.q_sb + (int64_t)qi * p.q_st +
                        (int64_t)h * p.q_sh;
          bulk_load(sQ + (stage * RMAX + lane) * D, qrow, Tr::kQRowBytes, &full[stage]);
        }
        if (lane < 2 * Tr::kStagePages && w < n) {
          const bool is_k = lane < Tr::kStagePages;
          T* dst = (is_k ? sK : sV) + (stage * Tr::kStagePages + w) * Tr::kPageElems;
          tma_load_4d(dst, is_k ? &tmk : &tmv, &full[stage], 0, g, c2, c3, pol);
        }
        if (++stage == Tr::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    // Drain: every issued stage must be consumed before the warp leaves, so
    // no bulk copy can still target this CTA's shared memory.
    if (lane == 0) {
      for (int i = 0; i < Tr::kStages; ++i) {
        if (!failed && !mbar_wait(&empty[stage], phase ^ 1)) failed = true;
        if (++stage == Tr::kStages) {
          stage = 0;
          phase ^= 1;
        }
      }
    }
    __syncwarp();
    return;
  }

  // ======================= consumers =======================
  int stage = 0;
  uint32_t phase = 0;
  bool failed = false;
  const int grp = lane >> 3;  // key slot within a QK pass
  const int sub = lane & 7;   // 16-byte chunk within the key row
  const int slot = warp % Tr::kStagePages;  // page of the stage this warp reads
  const int part = warp / Tr::kStagePages;  // which kPartKeys keys of that page

  for (int item = cta; item < num_items; item += num_ctas) {
    int b, g, s, nb, p0, p1;
    SeqInfo si;
    item_of(item, b, g, s, nb, p0, p1, si);
    const int R = si.qlen * p.G;  // <= RMAX for every item that exists
    const int kend = min(p1 * kPage, si.lk);

    // q rows -> registers (pre-scaled into the log2 domain) once the item's
    // first stage, which carries them, has landed
    float qf[RMAX][Tr::kQCh * 8];
    int lim[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      const int qi = r / p.G;
      lim[r] = p.causal ? qi + si.lk - si.qlen : 0x7fffffff;
#pragma unroll
      for (int e = 0; e < Tr::kQCh * 8; ++e) qf[r][e] = 0.f;
    }
    float m[RMAX], l[RMAX], o[RMAX][Tr::kPVE];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      m[r] = neg_inf();
      l[r] = 0.f;
#pragma unroll
      for (int e = 0; e < Tr::kPVE; ++e) o[r][e] = 0.f;
    }

    for (int pg = p0; pg < p1; pg += Tr::kStagePages) {
      if (!failed && !mbar_wait(&full[stage], phase)) {
        report(p.err, PA_DEVERR_TIMEOUT, b, pg);
        failed = true;
      }
      if (pg == p0) {
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          if (r < R) {
            const T* qrow = sQ + (stage * RMAX + r) * D;
#pragma unroll
            for (int c = 0; c < Tr::kQCh; ++c) {
              const uint4 u = *reinterpret_cast<const uint4*>(qrow + c * 64 + sub * 8);
              const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = E::to_f2(w4[e]);
                qf[r][c * 8 + 2 * e] = f.x * p.scale_log2;
                qf[r][c * 8 + 2 * e + 1] = f.y * p.scale_log2;
              }
            }
          }
        }
      }
      const int page = pg + slot;
      if (page < p1) {
        T* kp = sK + (stage * Tr::kStagePages + slot) * Tr::kPageElems;
        T* vp = sV + (stage * Tr::kStagePages + slot) * Tr::kPageElems;
        const int t_base = page * kPage;
        const int nvalid = min(kPage, kend - t_base);
        // New tokens among this warp's keys: patch the staged copy and append
        // them to the cache (each warp patches only the rows it reads).
        const int kb = part * Tr::kPartKeys;
        if (p.Lnew > 0 && t_base + min(nvalid, kb + Tr::kPartKeys) > si.old) {
          const int* info = sInfo + (stage * Tr::kStagePages + slot) * 3;
          const int c2 = info[0], c3 = info[1];
          const bool ok = info[2] != 0;
          const int t0 = max(si.old - t_base, kb);
          const int t1 = min(nvalid, kb + Tr::kPartKeys);
          constexpr int kChunks = D / 8;  // 16-byte chunks per row
          for (int idx = lane; idx < (t1 - t0) * kChunks; idx += 32) {
            const int t = t0 + idx / kChunks;
            const int c = idx % kChunks;
            const int64_t src = (((int64_t)b * p.Lnew + (t_base + t - si.old)) * p.Hkv + g) * D + c * 8;
            const uint4 kv = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.k_new) + src));
            const uint4 vv = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.v_new) + src));
            *reinterpret_cast<uint4*>(kp + t * D + c * 8) = kv;
            *reinterpret_cast<uint4*>(vp + t * D + c * 8) = vv;
            if (ok) {
              T* kdst = reinterpret_cast<T*>(p.k_cache) + (int64_t)c3 * p.k_sb +
                        (int64_t)(c2 + t) * p.k_st + (int64_t)g * p.k_sh + c * 8;
              T* vdst = reinterpret_cast<T*>(p.v_cache) + (int64_t)c3 * p.v_sb +
                        (int64_t)(c2 + t) * p.v_st + (int64_t)g * p.v_sh + c * 8;
              *reinterpret_cast<uint4*>(kdst) = kv;
              *reinterpret_cast<uint4*>(vdst) = vv;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
        }

        // ---- S = q K^T for this warp's keys of the page (passes of 4 keys)
        constexpr int kPasses = Tr::kPartKeys / 4;
        float sc[RMAX][kPasses];
#pragma unroll
        for (int ps = 0; ps < kPasses; ++ps) {
          const int t = kb + ps * 4 + grp;
          const T* krow = kp + t * D;
          float kf[Tr::kQCh * 8];
#pragma unroll
          for (int c = 0; c < Tr::kQCh; ++c) {
            const uint4 u = *reinterpret_cast<const uint4*>(krow + c * 64 + sub * 8);
            const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = E::to_f2(w4[e]);
              kf[c * 8 + 2 * e] = f.x;
              kf[c * 8 + 2 * e + 1] = f.y;
            }
          }
          const int kt = t_base + t;
#pragma unroll
          for (int r = 0; r < RMAX; ++r) {
            if (r < R) {
              float acc = 0.f;
#pragma unroll
              for (int e = 0; e < Tr::kQCh * 8; ++e) acc = fmaf(qf[r][e], kf[e], acc);
              acc += __shfl_xor_sync(0xffffffffu, acc, 1);
              acc += __shfl_xor_sync(0xffffffffu, acc, 2);
              acc += __shfl_xor_sync(0xffffffffu, acc, 4);
              const bool vis = (t < nvalid) && (kt <= lim[r]);
              sc[r][ps] = vis ? acc : neg_inf();
            }
          }
        }
        // ---- online softmax (log2 domain) and O += P V
        float pr[RMAX][kPasses];
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          if (r < R) {
            float mx = sc[r][0];
#pragma unroll
            for (int i = 1; i < kPasses; ++i) mx = fmaxf(mx, sc[r][i]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mnew = fmaxf(m[r], mx);
            float alpha = 1.f;
            if (mnew == neg_inf()) {
#pragma unroll
              for (int i = 0; i < kPasses; ++i) pr[r][i] = 0.f;
            } else {
              alpha = ex2(m[r] - mnew);
#pragma unroll
              for (int i = 0; i < kPasses; ++i) pr[r][i] = ex2(sc[r][i] - mnew);
            }
            float sum = pr[r][0];
#pragma unroll
            for (int i = 1; i < kPasses; ++i) sum += pr[r][i];
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            l[r] = l[r] * alpha + sum;
            m[r] = mnew;
#pragma unroll
            for (int e = 0; e < Tr::kPVE; ++e) o[r][e] *= alpha;
          }
        }
#pragma unroll
        for (int t = 0; t < Tr::kPartKeys; ++t) {
          if (kb + t < nvalid) {
            const T* vrow = vp + (kb + t) * D + lane * Tr::kPVE;
            float vf[Tr::kPVE];
            if constexpr (Tr::kPVE == 4) {
              const uint2 u = *reinterpret_cast<const uint2*>(vrow);
              const float2 a = E::to_f2(u.x), c = E::to_f2(u.y);
              vf[0] = a.x; vf[1] = a.y; vf[2] = c.x; vf[3] = c.y;
            } else {
              const uint32_t u = *reinterpret_cast<const uint32_t*>(vrow);
              const float2 a = E::to_f2(u);
              vf[0] = a.x; vf[1] = a.y;
            }
#pragma unroll
            for (int r = 0; r < RMAX; ++r) {
              if (r < R) {
                const float pt = __shfl_sync(0xffffffffu, pr[r][t >> 2], (t & 3) * 8);
#pragma unroll
                for (int e = 0; e < Tr::kPVE; ++e) o[r][e] = fmaf(pt, vf[e], o[r][e]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == Tr::kStages) {
        stage = 0;
        phase ^= 1;
      }
    }

    // ---- merge the four warps' partial softmax states
    constexpr int kRowF = D + 2;
    if (warp > 0) {
      float* dst = sMerge + (warp - 1) * RMAX * kRowF;
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        if (r < R) {
#pragma unroll
          for (int e = 0; e < Tr::kPVE; ++e) dst[r * kRowF + lane * Tr::kPVE + e] = o[r][e];
          if (lane == 0) {
            dst[r * kRowF + D] = m[r];
            dst[r * kRowF + D + 1] = l[r];
          }
        }
      }
    }
    named_barrier(1, Tr::kConsumerWarps * 32);
    if (warp == 0) {
      const bool to_partial = nb > 1;
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        if (r < R) {
          float M = m[r];
          for (int w = 1; w < Tr::kConsumerWarps; ++w)
            M = fmaxf(M, sMerge[(w - 1) * RMAX * kRowF + r * kRowF + D]);
          float L = 0.f;
          float acc[Tr::kPVE];
          if (M == neg_inf()) {
#pragma unroll
            for (int e = 0; e < Tr::kPVE; ++e) acc[e] = 0.f;
          } else {
            const float a0 = ex2(m[r] - M);
            L = l[r] * a0;
#pragma unroll
            for (int e = 0; e < Tr::kPVE; ++e) acc[e] = o[r][e] * a0;
            for (int w = 1; w < Tr::kConsumerWarps; ++w) {
              const float* src = sMerge + (w - 1) * RMAX * kRowF + r * kRowF;
              const float aw = ex2(src[D] - M);
              L += src[D + 1] * aw;
#pragma unroll
              for (int e = 0; e < Tr::kPVE; ++e) acc[e] = fmaf(src[lane * Tr::kPVE + e], aw, acc[e]);
            }
          }
          const float inv = (L > 0.f) ? 1.f / L : 0.f;
          const float lse_v = (L > 0.f) ? (M + lg2(L)) * kLn2 : neg_inf();
          const int qi = r / p.G;
          const int h = g * p.G + (r % p.G);
          const int64_t row = si.row0 + qi;  // global row index
          if (to_partial) {
            float* op = p.o_part + (((int64_t)s * (p.cu_seqlens_q ? p.total_q : (int64_t)p.B * p.Lq) + row) * p.Hq + h) * D;
#pragma unroll
            for (int e = 0; e < Tr::kPVE; ++e) op[lane * Tr::kPVE + e] = acc[e] * inv;
            if (lane == 0)
              p.lse_part[((int64_t)s * (p.cu_seqlens_q ? p.total_q : (int64_t)p.B * p.Lq) + row) * p.Hq + h] = lse_v;
          } else {
            T* orow = reinterpret_cast<T*>(p.out) + (row * p.Hq + h) * D + lane * Tr::kPVE;
            if constexpr (Tr::kPVE == 4) {
              uint2 u;
              u.x = E::from_f2(acc[0] * inv, acc[1] * inv);
              u.y = E::from_f2(acc[2] * inv, acc[3] * inv);
              *reinterpret_cast<uint2*>(orow) = u;
            } else {
              *reinterpret_cast<uint32_t*>(orow) = E::from_f2(acc[0] * inv, acc[1] * inv);
            }
            if (p.lse != nullptr && lane == 0) {
              if (p.cu_seqlens_q != nullptr)
                p.lse[(int64_t)h * p.total_q + row] = lse_v;
              else
                p.lse[((int64_t)b * p.Hq + h) * p.Lq + qi] = lse_v;
            }
          }
        }
      }
    }
    named_barrier(1, Tr::kConsumerWarps * 32);
  }
}

template <int D, typename T, int RMAX>
cudaError_t launch_t(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                     cudaStream_t st) {
  using Tr = DecodeTraits<D, T, RMAX>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, T, RMAX>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Tr::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int grid = p.grid_ctas;
  long long max_items;
  if (p.s_max <= 1 && p.cu_seqlens_q == nullptr)
    max_items = (long long)p.B * p.Hkv;
  else
    max_items = (long long)p.B * p.Hkv * (p.s_max < 1 ? 1 : p.s_max);
  if (max_items < grid) grid = (int)max_items;
  if (grid < 1) grid = 1;
  decode_kernel<D, T, RMAX><<<grid, Tr::kThreads, Tr::kSmemBytes, st>>>(p, tmk, tmv);
  return cudaGetLastError();
}

template <int D, typename T, int RMAX>
int occupancy_t() {
  using Tr = DecodeTraits<D, T, RMAX>;
  if (cudaFuncSetAttribute(decode_kernel<D, T, RMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           Tr::kSmemBytes) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, T, RMAX>, Tr::kThreads,
                                                    Tr::kSmemBytes) != cudaSuccess)
    return 0;
  return n;
}

template <int D, typename T>
cudaError_t launch_r(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                     int rmax, cudaStream_t st) {
  switch (rmax) {
    case 1: return launch_t<D, T, 1>(p, tmk, tmv, st);
    case 2: return launch_t<D, T, 2>(p, tmk, tmv, st);
  }
  return cudaErrorInvalidValue;
}

template <int D, typename T>
int occ_r(int rmax) {
  switch (rmax) {
    case 1: return occupancy_t<D, T, 1>();
    case 2: return occupancy_t<D, T, 2>();
  }
  return 0;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& tmk, const CUtensorMap& tmv,
                          int D, int dtype, int rmax, cudaStream_t st) {
  if (D == 128 && dtype == PA_F16) return launch_r<128, __half>(p, tmk, tmv, rmax, st);
  if (D == 128 && dtype == PA_BF16) return launch_r<128, __nv_bfloat16>(p, tmk, tmv, rmax, st);
  if (D == 64 && dtype == PA_F16) return launch_r<64, __half>(p, tmk, tmv, rmax, st);
  if (D == 64 && dtype == PA_BF16) return launch_r<64, __nv_bfloat16>(p, tmk, tmv, rmax, st);
  return cudaErrorInvalidValue;
}

int decode_ctas_per_sm(int D, int dtype, int rmax) {
  if (D == 128 && dtype == PA_F16) return occ_r<128, __half>(rmax);
  if (D == 128 && dtype == PA_BF16) return occ_r<128, __nv_bfloat16>(rmax);
  if (D == 64 && dtype == PA_F16) return occ_r<64, __half>(rmax);
  if (D == 64 && dtype == PA_BF16) return occ_r<64, __nv_bfloat16>(rmax);
  return 0;
}

}  // namespace pa
