// Persistent tensor-core attention engine over a paged KV cache (sm_103a).
//
// One launch walks a work list that every CTA derives on the GPU from the
// sequence lengths (no host read of lengths: flash-attention #1000
// "Inappropriate Number of Splits ...").  Two kinds of items:
//   kind 0  a 128-row query tile of ONE query head (long prefills): keys
//           [0, causal limit of the tile) -- the flash_attn_with_kvcache
//           prefill of flash-attention #824 "Add support for small page sizes".
//   kind 1  the q_len * G query rows (<= 128) of ALL G query heads that share
//           one kv head, packed into one tile (GQA packing: K/V streamed once
//           per kv head), against one split of the keys; split outputs go to
//           partials that the combine kernel merges -- decode, multi-query
//           decode and short chunked prefills.
// A varlen batch may mix both kinds in one launch: the unified launch of vLLM
// #6052 "Unify the kernel used in flash attention backend".
// Dealing: uniform calls without splits round-robin; varlen batches a
// contiguous run of units of equal estimated cost per CTA; kvcache packed
// calls with automatic splits (the TB instantiation) an equal share of the
// concatenated streams' key tiles per CTA, cutting streams at the share
// boundaries (split counts then kept per stream).
//
// CTA = 512 threads (16 warps), one per SM, persistent over items:
//   warps 0-7  softmax: warps w and w+4 share tile rows 32(w%4).. (their TMEM
//              lane quarter), each taking 64 of the 128 columns.  S from TMEM,
//              masking, running max / sum in the log2 domain, P (fp16/bf16)
//              written back over S in TMEM, lazy O rescale (only when the max
//              grows by more than 2^8), epilogue.
//   warps 8-11 TMA producers: Q of the item (warp 8), then per 128-key tile
//              8 pages of K (warps 8-9) and of V (warps 10-11), each page
//              resolved absolutely from the block table.
//   warps 12-13 idle: they only place the issuers below on the schedulers
//              (warp % 4) of the V producers, away from the K producers'.
//   warp 14    TMEM owner and P V issuer: O += P V with P read from TMEM.
//   warp 15    Q K^T issuer: copies each item's Q into TMEM (tcgen05.cp), then
//              S = Q K^T with Q from TMEM and K from shared memory into one of
//              NB TMEM buffers, tile t once P V of tile t-NB (whose P occupies
//              the buffer) has completed.
// TMEM: S/P of tile t in cols [128 (t % NB), +128), then O (D columns), then
// Q (D / 2 columns); NB = 2 for head dim 128, 3 for 64.
// Pipeline state (stage and buffer parities) runs on across items.
#include <type_traits>

#include "pa_common.cuh"
#include "pa_engine.h"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kBM = 128;                 // tile rows
constexpr int kBN = 128;                 // keys per KV tile
constexpr int kTilePages = kBN / kPage;  // 8
// S/P buffers in TMEM (128 columns each; O and then Q follow them).  Q K^T of
// tile t reuses the buffer of tile t - NB once P V of that tile has
// completed, so the chain softmax(t) -> P V(t) -> Q K^T(t+NB) -> softmax(t+NB)
// spans NB tiles.  Buffer of tile t: t mod NB; barrier phase parity (t / NB) mod 2.
template <int NB> __device__ __forceinline__ int sbuf_of(int t) { return t % NB; }
template <int NB> __device__ __forceinline__ uint32_t sbuf_par_of(int t) {
  return (uint32_t)((t / NB) & 1);
}
constexpr float kRescaleThreshold = 8.0f;
// Cost of one work item beyond its key tiles, in tiles (epilogue and the next
// item's set-up: about 5600 SM cycles against about 2800 per tile, plus the Q
// load; 3 measured best among 1-4 on the mixed batches).
constexpr int kItemTiles = 3;
constexpr int kSoftWarps = 8;               // softmax warps (two per TMEM lane quarter)
constexpr int kProdWarps = 4;               // TMA producer warps (issue throughput is per warp)
constexpr int kWarpTMA = kSoftWarps;        // first TMA producer warp
// Warps 12 and 13 do nothing: with 16 warps the two MMA issuers land on the
// schedulers of warps 2/6/10 and 3/7/11 (measured: +5 % prefill throughput
// over issuers on the schedulers shared with warps 0/4/8 and 1/5/9).
constexpr int kWarpMMA = kSoftWarps + kProdWarps + 2;  // P V issuer + TMEM owner
constexpr int kWarpQK = kWarpMMA + 1;               // Q K^T issuer
constexpr int kThreads = (kSoftWarps + kProdWarps + 4) * 32;

template <int D>
struct EngTraits {
  static constexpr int kHalves = D / 64;
  static constexpr int kSlab = 128 * 128;  // one 128-row x 128-byte slab
  static constexpr int kStages = (D == 128) ? 2 : 3;
  // TMEM: kSBufs S/P buffers of 128 columns, O (D columns), Q (D / 2 columns:
  // two 16-bit values per column) -- 2 x 128 + 128 + 64 = 448 for head dim
  // 128, 3 x 128 + 64 + 32 = 480 for 64, of 512.
  static constexpr int kSBufs = (D == 128) ? 2 : 3;
  static constexpr int kQBytes = kHalves * kSlab;
  static constexpr int kKVBytes = kHalves * kSlab;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffPre = kOffV + kStages * kKVBytes;  // two int[kEngineMaxB + 1] prefix sums
  static constexpr int kOffBar = kOffPre + ((2 * (kEngineMaxB + 1) * 4 + 15) & ~15);
  static constexpr int kNumBars = 2 + 4 * kStages + 3 * kSBufs + 1 + 1;
  static_assert(kSBufs * 128 + D + D / 2 <= 512, "TMEM columns");
  // With two stages a K stage is free exactly when Q K^T of the tile two back
  // has completed, which s_full of that parity already signals; likewise a V
  // stage and pv_done.  The producers then wait on those, and the MMA thread
  // saves two commits per tile.
  static constexpr bool kSharedEmpty = kStages == 2;
  static constexpr int kOffX = (kOffBar + kNumBars * 8 + 15) & ~15;  // row max / sum exchange
  static constexpr int kOffMisc = kOffX + (2 * 2 * 128 + 128) * 4;
  static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
  static constexpr uint32_t kTmemCols = 512;
};

struct SeqI {
  int qlen, lk;
  int64_t row0;  // global row index of query 0 (output / partial addressing)
  int qcoord;    // TMA row coordinate of query 0
  int qb;        // TMA batch coordinate
};

__device__ __forceinline__ SeqI seq_of(const EngineParams& p, int b, bool rep) {
  SeqI s;
  int old;
  if (p.cu_seqlens_q != nullptr) {
    const int q0 = __ldg(p.cu_seqlens_q + b);
    s.qlen = __ldg(p.cu_seqlens_q + b + 1) - q0;
    s.lk = __ldg(p.seqlens_k + b);
    old = s.lk;
    s.row0 = q0;
    s.qcoord = q0;
    s.qb = 0;
  } else {
    s.qlen = p.Lq;
    old = __ldg(p.cache_seqlens + b);
    s.lk = old + p.Lnew;
    s.row0 = (int64_t)b * p.Lq;
    s.qcoord = 0;
    s.qb = b;
  }
  bool bad = old < 0 || s.lk < 0 || s.lk > p.max_seqlen_k || s.qlen < 0;
  if (p.block_table != nullptr)
    bad = bad || (((int64_t)(s.lk + kPage - 1) / kPage + (1 << p.page_shift) - 1) >> p.page_shift) >
                     p.max_pages;
  else
    bad = bad || (int64_t)s.lk > p.extent;
  if (bad) {
    if (rep) report(p.err, PA_DEVERR_LENGTH, b, s.qlen < 0 ? s.qlen : s.lk);
    s.lk = 0;
    if (s.qlen < 0) s.qlen = 0;
  }
  return s;
}

__device__ __forceinline__ bool packed_seq(const EngineParams& p, int qlen) {
  return qlen > 0 && qlen * p.G <= p.pack_rows;
}

// Pages per split of a packed sequence (a multiple of one 8-page KV tile) and
// the split count.
__device__ __forceinline__ int packed_split(const EngineParams& p, int pages, int chunk,
                                            int* n_out) {
  if (p.s_max <= 1 || pages <= 0) {
    *n_out = 1;
    return pages > 0 ? pages : 0;
  }
  int n = (pages + chunk - 1) / chunk;
  n = max(1, min(n, p.s_max));
  int per = (pages + n - 1) / n;
  per = (per + kTilePages - 1) / kTilePages * kTilePages;
  *n_out = (pages + per - 1) / per;
  return per;
}

struct Item {
  int kind, b, head, qs, nrows, qlen, lk, k0, k1, ntiles, split, nsplit;
  int64_t row0;
  int qcoord, qb;
};

struct Sched {
  bool uniform;   // kvcache call: every sequence has the same query length
  bool packed_u;  // uniform and packed
  // tile-granular shares (the engine's TB instantiation, EngineParams::
  // tilebal): chunk is the share and total1 the positions; CTA c takes
  // positions [c * share, (c + 1) * share)
  int total0, total1, chunk;
  const int* pre0;
  const int* pre1;
};

// Key tiles a stream of `lk` keys occupies in the tile-granular position
// space: its tiles, or one position for a stream without keys (so that
// exactly one CTA owns it and writes its empty output).
__device__ __forceinline__ int tb_span(int lk) { return lk > 0 ? (lk + kBN - 1) / kBN : 1; }

__device__ __forceinline__ int last_le(const int* pre, int n, int x) {
  int lo = 0, hi = n;  // last index in [0, n) with pre[idx] <= x
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

// Work unit `idx`, sub-item u (0 or 1).  A kind-0 unit is a PAIR of query
// tiles of one head, t and q_tiles-1-t (heaviest with lightest under causal
// masking), so every unit costs about the same: CTAs walking units
// round-robin stay in step, and the query tiles of a head stream its K/V
// through L2 together.  Kind-1 units have one item; their second sub-item (and
// the second of an odd middle pair) is empty (kind -1, no rows, no tiles).
// Work units are (item index idx, half u) pairs, wu = 2 idx + u, dealt to the
// CTAs by idx (the dealing note at the top of this file).  A kind-0 index
// carries a pair of query tiles (u = 0 and 1); a packed index only u = 0, so
// its u = 1 half is skipped from the schedule alone, without looking the unit
// up (every role skips alike).
__device__ __forceinline__ bool empty_half(const Sched& sc, int wu) {
  return (wu & 1) && (sc.uniform ? sc.packed_u : (wu >> 1) >= sc.total0);
}

template <bool TB>
__device__ __forceinline__ Item get_item(const EngineParams& p, const Sched& sc, int idx, int u) {
  Item it;
  if constexpr (TB) {
    // stream idx = (sequence, kv head); its piece inside this CTA's positions
    const int b = idx / p.Hkv;
    it.b = b;
    it.head = idx - b * p.Hkv;
    const SeqI q = seq_of(p, b, true);
    it.qlen = q.qlen;
    it.lk = q.lk;
    it.row0 = q.row0;
    it.qcoord = q.qcoord;
    it.qb = q.qb;
    it.qs = 0;
    const int span = tb_span(q.lk);
    const int P = sc.pre1[b] + it.head * span;
    const int share = sc.chunk;
    const int lo = (int)min((long long)sc.total1, (long long)blockIdx.x * share);
    const int hi = min(sc.total1, lo + share);
    const int x0 = max(lo, P), x1 = min(hi, P + span);
    if (u != 0 || !packed_seq(p, q.qlen) || x0 >= x1) {
      it.kind = -1;
      it.nrows = 0;
      it.k0 = it.k1 = 0;
      it.split = 0;
      it.nsplit = 1;
      it.ntiles = 0;
      return it;
    }
    it.kind = 1;
    it.nrows = q.qlen * p.G;
    it.split = x0 / share - P / share;
    it.nsplit = (P + span - 1) / share - P / share + 1;
    it.k0 = min((x0 - P) * kBN, q.lk);
    it.k1 = min((x1 - P) * kBN, q.lk);
    it.ntiles = it.k1 > it.k0 ? (it.k1 - it.k0 + kBN - 1) / kBN : 0;
    return it;
  }
  int b, head, t = 0, s = 0;
  bool packed, null_item = false;
  auto pick_pair = [&](int qt, int pi) {
    t = (u == 0) ? qt - 1 - pi : pi;
    null_item = (u == 1 && pi == qt - 1 - pi);
  };
  if (sc.uniform) {
    packed = sc.packed_u;
    if (packed) {
      const int per_b = p.Hkv * max(1, p.s_max);
      b = idx / per_b;
      const int li = idx % per_b;
      s = li / p.Hkv;
      head = li % p.Hkv;
      null_item = u == 1;
    } else {
      const int qt = p.max_q_tiles;
      const int pp = (qt + 1) / 2;
      const int bh = idx / pp;
      pick_pair(qt, idx % pp);
      b = bh / p.Hq;
      head = bh % p.Hq;
    }
  } else if (idx < sc.total0) {
    packed = false;
    b = last_le(sc.pre0, p.B, idx);
    const int li = idx - sc.pre0[b];
    const SeqI q = seq_of(p, b, false);
    const int qt = (q.qlen + kBM - 1) / kBM;
    const int pp = (qt + 1) / 2;
    head = li / pp;
    pick_pair(qt, li % pp);
  } else {
    packed = true;
    const int i1 = idx - sc.total0;
    b = last_le(sc.pre1, p.B, i1);
    const int li = i1 - sc.pre1[b];
    s = li / p.Hkv;
    head = li % p.Hkv;
    null_item = u == 1;
  }
  const SeqI q = seq_of(p, b, true);
  it.b = b;
  it.head = head;
  it.qlen = q.qlen;
  it.lk = q.lk;
  it.row0 = q.row0;
  it.qcoord = q.qcoord;
  it.qb = q.qb;
  if (null_item) {
    it.kind = -1;
    it.qs = 0;
    it.nrows = 0;
    it.k0 = it.k1 = 0;
    it.split = 0;
    it.nsplit = 1;
  } else if (!packed) {
    it.kind = 0;
    it.qs = t * kBM;
    it.nrows = max(0, min(kBM, q.qlen - it.qs));
    it.k0 = 0;
    int k1 = q.lk;
    if (p.causal) k1 = min(q.lk, it.qs + it.nrows + q.lk - q.qlen);
    it.k1 = max(0, k1);
    if (it.nrows == 0) it.k1 = 0;
    it.split = 0;
    it.nsplit = 1;
  } else {
    it.kind = 1;
    it.qs = 0;
    it.nrows = q.qlen * p.G;
    const int pages = (q.lk + kPage - 1) / kPage;
    int n;
    const int per = packed_split(p, pages, sc.chunk, &n);
    it.split = s;
    it.nsplit = n;
    it.k0 = min(s * per * kPage, q.lk);
    it.k1 = min((s + 1) * per * kPage, q.lk);
    if (s >= n) it.k1 = it.k0;  // uniform mode: splits past this sequence's count are empty
  }
  it.ntiles = it.k1 > it.k0 ? (it.k1 - it.k0 + kBN - 1) / kBN : 0;
  return it;
}

// TB: the tile-granular schedule of kvcache packed calls with automatic
// splits (a separate instantiation, so that the other calls' role loops carry
// none of its code at the kernel's register cap).
template <int D, typename T, bool TB>
__global__ void __launch_bounds__(kThreads, 1)
    engine_kernel(const EngineParams p, const __grid_constant__ CUtensorMap tm_q1,
                  const __grid_constant__ CUtensorMap tm_q2,
                  const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v) {
  using Tr = EngTraits<D>;
  constexpr int kSBufs = Tr::kSBufs;
  auto sbuf = [](int t) { return sbuf_of<Tr::kSBufs>(t); };
  auto sbuf_par = [](int t) { return sbuf_par_of<Tr::kSBufs>(t); };
  using E = Elem<T>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + Tr::kOffQ;
  uint8_t* sK = smem + Tr::kOffK;
  uint8_t* sV = smem + Tr::kOffV;
  int* pre0 = reinterpret_cast<int*>(smem + Tr::kOffPre);
  int* pre1 = pre0 + (kEngineMaxB + 1);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Tr::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* v_full = k_full + Tr::kStages;
  uint64_t* k_empty = v_full + Tr::kStages;
  uint64_t* v_empty = k_empty + Tr::kStages;
  uint64_t* s_full = v_empty + Tr::kStages;  // [kSBufs], tile t -> t % kSBufs
  // [kSBufs] by S buffer: the softmax warps are synchronised only in pairs,
  // so one lane quarter may arrive for tile t+1 or t+2 before another has
  // arrived for tile t (t+3 needs P V of t); one barrier per buffer keeps
  // those arrivals apart.
  uint64_t* p_full = s_full + kSBufs;
  uint64_t* pv_done = p_full + kSBufs;  // [kSBufs]: P V of a tile of that buffer completed
  uint64_t* o_free = pv_done + kSBufs;
  uint64_t* mma_fin = o_free + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + Tr::kOffMisc);
  int* misc = reinterpret_cast<int*>(smem + Tr::kOffMisc + 16);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < Tr::kStages; ++i) {
      mbar_init(&k_full[i], kProdWarps / 2);
      mbar_init(&v_full[i], kProdWarps / 2);
      mbar_init(&k_empty[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < kSBufs; ++i) mbar_init(&s_full[i], 1);
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(&p_full[i], kSoftWarps);
      mbar_init(&pv_done[i], 1);
    }
    mbar_init(o_free, kSoftWarps);
    mbar_init(mma_fin, 2);  // one commit from each MMA issuer
    fence_mbar_init();
  }
  if (warp == kWarpMMA) {
    tc::tmem_alloc(tslot, Tr::kTmemCols);
    tc::tmem_relinquish();
  }

  // ---- device schedule
  Sched sc;
  int unit_first = 0, unit_end = 0;  // varlen: this CTA's contiguous run of units
  sc.uniform = p.cu_seqlens_q == nullptr && (p.s_max <= 1 || !(p.Lq > 0 && p.Lq * p.G <= p.pack_rows));
  sc.packed_u = p.cu_seqlens_q == nullptr && p.Lq > 0 && p.Lq * p.G <= p.pack_rows;
  sc.pre0 = pre0;
  sc.pre1 = pre1;
  sc.chunk = 0;
  if (sc.uniform) {
    sc.total0 = sc.packed_u ? 0 : p.B * p.Hq * ((p.max_q_tiles + 1) / 2);
    sc.total1 = sc.packed_u ? p.B * p.Hkv * max(1, p.s_max) : 0;
  } else {
    long long part = 0;
    for (int b = tid; b < p.B; b += kThreads) {
      const SeqI q = seq_of(p, b, true);
      if (packed_seq(p, q.qlen)) part += (q.lk + kPage - 1) / kPage;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    long long* red = reinterpret_cast<long long*>(sV);  // V is free before the first tile
    if (lane == 0) red[warp] = part;
    __syncthreads();
    long long total = 0;
    for (int w = 0; w < kThreads / 32; ++w) total += red[w];
    {
      long long slots = (long long)p.target_ctas;
      long long c = (total * p.Hkv + slots - 1) / max(1LL, slots);
      if (c < p.min_chunk_pages) c = p.min_chunk_pages;
      if (c > (1 << 28)) c = 1 << 28;
      sc.chunk = (int)((c + kTilePages - 1) / kTilePages * kTilePages);
    }
    __syncthreads();
    // cost prefixes over the same unit order, in key tiles (scratch in the
    // K stages, free before the first tile): varlen batches deal every CTA a
    // contiguous run of units of equal estimated cost (see wu_first below)
    int* cp0 = reinterpret_cast<int*>(sK);
    int* cp1 = cp0 + (kEngineMaxB + 1);
    if (warp == 0) {
      int carry0 = 0, carry1 = 0, ccarry0 = 0, ccarry1 = 0;
      for (int base = 0; base < p.B; base += 32) {
        const int b = base + lane;
        int c0 = 0, c1 = 0, w0 = 0, w1 = 0;
        if (b < p.B) {
          const SeqI q = seq_of(p, b, false);
          int n = 0;
          if (TB && packed_seq(p, q.qlen)) {
            c1 = p.Hkv * tb_span(q.lk);  // key-tile positions of the sequence's streams
          } else if (packed_seq(p, q.qlen)) {
            const int per = packed_split(p, (q.lk + kPage - 1) / kPage, sc.chunk, &n);
            c1 = n * p.Hkv;
            w1 = c1 * ((per + kTilePages - 1) / kTilePages + kItemTiles);
          } else if (q.qlen > 0) {
            const int qt = (q.qlen + kBM - 1) / kBM;
            const int pairs = (qt + 1) / 2;
            c0 = pairs * p.Hq;
            // key tiles of all query tiles of one head, shared out over its
            // pairs (the pairing makes them about equal)
            int tiles = 0;
            for (int t = 0; t < qt; ++t) {
              const int qs = t * kBM, nrows = min(kBM, q.qlen - qs);
              int k1 = q.lk;
              if (p.causal) k1 = min(q.lk, qs + nrows + q.lk - q.qlen);
              tiles += (max(0, k1) + kBN - 1) / kBN;
            }
            w0 = c0 * ((tiles + pairs - 1) / pairs + 2 * kItemTiles);
          }
          // split count read by the combine step, for EVERY sequence: 0 for
          // sequences written directly (unsplit, query tiles, empty entries)
          if (!TB && blockIdx.x == 0 && p.nsplit != nullptr) p.nsplit[b] = n > 1 ? n : 0;
        }
        int i0 = c0, i1 = c1, j0 = w0, j1 = w1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y0 = __shfl_up_sync(0xffffffffu, i0, o);
          const int y1 = __shfl_up_sync(0xffffffffu, i1, o);
          const int z0 = __shfl_up_sync(0xffffffffu, j0, o);
          const int z1 = __shfl_up_sync(0xffffffffu, j1, o);
          if (lane >= o) {
            i0 += y0;
            i1 += y1;
            j0 += z0;
            j1 += z1;
          }
        }
        if (b < p.B) {
          pre0[b] = carry0 + i0 - c0;
          pre1[b] = carry1 + i1 - c1;
          cp0[b] = ccarry0 + j0 - w0;
          cp1[b] = ccarry1 + j1 - w1;
        }
        carry0 += __shfl_sync(0xffffffffu, i0, 31);
        carry1 += __shfl_sync(0xffffffffu, i1, 31);
        ccarry0 += __shfl_sync(0xffffffffu, j0, 31);
        ccarry1 += __shfl_sync(0xffffffffu, j1, 31);
      }
      if (lane == 0) {
        pre0[p.B] = carry0;
        pre1[p.B] = carry1;
        cp0[p.B] = ccarry0;
        cp1[p.B] = ccarry1;
        misc[0] = carry0;
        misc[1] = carry1;
      }
    }
    __syncthreads();
    sc.total0 = misc[0];
    sc.total1 = misc[1];
    if constexpr (TB) {
      // Tile-granular shares: the (sequence, kv head) streams' key tiles laid
      // end to end (pre1: positions before each sequence), every CTA takes
      // `share` consecutive positions, and a stream cut by a share boundary
      // runs as split pieces that the combine step merges.  The share is at
      // least a capacity stream over s_max - 1, so no stream has more than
      // s_max pieces.
      const int W = sc.total1;
      const int tcap = tb_span(p.max_seqlen_k);
      int share = (W + (int)gridDim.x - 1) / (int)gridDim.x;
      if (p.s_max > 1) share = max(share, (tcap + p.s_max - 2) / (p.s_max - 1));
      share = max(share, 1);
      sc.chunk = share;
      const int lo = (int)min((long long)W, (long long)blockIdx.x * share);
      const int hi = min(W, lo + share);
      auto stream_at = [&](int x) {
        const int b = last_le(pre1, p.B, x);
        return b * p.Hkv + (x - pre1[b]) / tb_span(seq_of(p, b, false).lk);
      };
      unit_first = lo < hi ? stream_at(lo) : 0;
      unit_end = lo < hi ? stream_at(hi - 1) + 1 : 0;
      if (blockIdx.x == 0 && p.nsplit != nullptr) {
        // pieces per stream, read by the combine step (0: written directly)
        for (int i = tid; i < p.B * p.Hkv; i += kThreads) {
          const int b = i / p.Hkv;
          const SeqI q = seq_of(p, b, false);
          int n = 0;
          if (packed_seq(p, q.qlen)) {
            const int span = tb_span(q.lk);
            const int P0 = pre1[b] + (i - b * p.Hkv) * span;
            n = (P0 + span - 1) / share - P0 / share + 1;
          }
          p.nsplit[i] = n > 1 ? n : 0;
        }
      }
    } else {
      // this CTA's units: those whose cost position (the cost of all units
      // before them) lies in [cta * share, (cta + 1) * share)
      const long long wtot = (long long)cp0[p.B] + cp1[p.B];
      const long long wshare = (wtot + gridDim.x - 1) / gridDim.x;
      auto unit_at = [&](long long x) -> int {
        if (x >= wtot) return sc.total0 + sc.total1;
        const bool k0 = x < cp0[p.B];
        const int* cp = k0 ? cp0 : cp1;
        const int* pre = k0 ? pre0 : pre1;
        const int xi = (int)(k0 ? x : x - cp0[p.B]);
        const int b = last_le(cp, p.B, xi);
        const int n = pre[b + 1] - pre[b];
        const int u = n > 0 ? (cp[b + 1] - cp[b]) / n : 0;
        const int li = u > 0 ? (xi - cp[b] + u - 1) / u : 0;
        return (k0 ? 0 : sc.total0) + pre[b] + min(li, n);
      };
      unit_first = unit_at((long long)blockIdx.x * wshare);
      unit_end = unit_at((long long)(blockIdx.x + 1) * wshare);
    }
  }
  // the combine grid that follows may be scheduled now; it waits on the
  // device for this grid's completion before reading any partial
  griddep_launch_dependents();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tbase = *tslot;
  const uint32_t tO = tbase + kSBufs * 128;
  const uint32_t tQ = tO + D;  // Q of the current item, copied from shared memory
  auto tS = [&](int t) { return tbase + (uint32_t)(sbuf(t) * 128); };
  const int total = sc.total0 + sc.total1;
  // Work-unit halves of this CTA: uniform batches (equal units) deal units
  // round-robin; varlen batches take the CTA's contiguous run of units of
  // equal estimated cost, so that sequences of different lengths do not pile
  // up on some CTAs (measured round-robin: average / slowest CTA busy time
  // 0.83 and 0.73 on the 32 x 128 and 12 x 64 mixed batches).
  const bool ranged = !sc.uniform;
  const int wu_first = ranged ? 2 * unit_first : 2 * (int)blockIdx.x;
  const int wu_end = ranged ? 2 * unit_end : 2 * total;
  auto wu_next = [&](int wu) {
    return (ranged || !(wu & 1)) ? wu + 1 : wu + 2 * (int)gridDim.x - 1;
  };

  if (warp >= kWarpTMA && warp < kWarpTMA + kProdWarps) {
    // ======================= TMA producers =======================
    // Warps 0 and 1 of the group load K tiles, warps 2 and 3 V tiles, each
    // taking alternate pages of every tile (TMA issue throughput grows with
    // the number of issuing warps) and arriving on the stage barrier with its
    // share of the bytes.  K and V run independently: a K stage is refilled as
    // soon as Q K^T has read it, without waiting behind the V stage, which
    // frees only after P V at the end of the tile's chain.
    // Within a warp:  Block-table entries are loaded 32 pages
    // (4 KV tiles) at a time, one lane per page, a batch ahead of use and with
    // no dependent instruction until the tile is issued, so the table reads
    // never sit on the copy path; every entry is validated when used.  Lane 0
    // waits for free stages and issues the copies.
    const uint64_t pol_kv = l2_policy_evict_last();
    const uint64_t pol_q = l2_policy_evict_first();
    const bool paged = p.block_table != nullptr;
    const int pw = warp - kWarpTMA;
    const bool is_v = pw >= kProdWarps / 2;
    const int sub = pw % (kProdWarps / 2);
    uint64_t* x_full = is_v ? v_full : k_full;
    uint64_t* x_empty = is_v ? v_empty : k_empty;
    // with two stages, stage of tile t is free once Q K^T (K) or P V (V) of
    // tile t-2 has completed: s_full / pv_done of that tile
    uint64_t* x_done = is_v ? pv_done : s_full;
    uint8_t* sX = is_v ? sV : sK;
    const CUtensorMap* tm_x = is_v ? &tm_v : &tm_k;
    bool failed = false;
    int tctr = 0, a = 0;
    int issued = 0, q_issued = 0;  // tiles (and items' Q) whose copies were issued
    for (int wu = wu_first; wu < wu_end; wu = wu_next(wu)) {
      if (empty_half(sc, wu)) continue;
      const Item it = get_item<TB>(p, sc, wu >> 1, wu & 1);
      if (it.ntiles == 0) continue;
      const int g = it.kind == 0 ? it.head / p.G : it.head;
      const int pg_begin = it.k0 / kPage;
      const int pg_end = (it.k1 + kPage - 1) / kPage;
      const int32_t* trow = paged ? p.block_table + (int64_t)it.b * p.bt_stride : nullptr;
      // raw table entry of 16-token box pg_begin + 32*batch + lane (its page:
      // entry box >> page_shift)
      auto load_batch = [&](int batch) -> int {
        const int lp = pg_begin + 32 * batch + lane;
        const int entry = lp >> p.page_shift;
        return (paged && lp < pg_end && entry < p.max_pages) ? __ldg(trow + entry) : 0;
      };
      int cur = load_batch(0);
      int nxt = (it.ntiles > 4) ? load_batch(1) : 0;
      if (pw == 0 && lane == 0) {
        if (a >= 1 && !failed && !mbar_wait(q_empty, (uint32_t)((a - 1) & 1))) {
          report(p.err, PA_DEVERR_TIMEOUT, it.b, -1);
          failed = true;
        }
        if (!failed) {
          mbar_arrive_expect_tx(q_full, Tr::kQBytes);
          for (int hh = 0; hh < Tr::kHalves; ++hh) {
            if (it.kind == 0)
              tma_load_4d(sQ + hh * Tr::kSlab, &tm_q1, q_full, hh * 64, it.head,
                          it.qcoord + it.qs, it.qb, pol_q);
            else
              tma_load_4d(sQ + hh * Tr::kSlab, &tm_q2, q_full, hh * 64, it.head * p.G,
                          it.qcoord, it.qb, pol_q);
          }
          q_issued = a + 1;
        }
      }
      __syncwarp();
      for (int j = 0; j < it.ntiles; ++j) {
        if (j > 0 && (j & 3) == 0) {
          cur = nxt;
          nxt = (j + 4 < it.ntiles) ? load_batch((j >> 2) + 1) : 0;
        }
        const int Tj = tctr + j;
        const int s = Tj % Tr::kStages;
        const uint32_t par = (uint32_t)((Tj / Tr::kStages) & 1);
        const int pg0 = pg_begin + j * kTilePages;
        const int npg = min(kTilePages, pg_end - pg0);
        int c2[kTilePages], c3[kTilePages];
#pragma unroll
        for (int i = 0; i < kTilePages; ++i) {
          const int raw = __shfl_sync(0xffffffffu, cur, (j & 3) * kTilePages + i);
          const int lp = pg0 + i;
          bool ok;
          if (paged) {
            ok = (lp >> p.page_shift) < p.max_pages && raw >= 0 && (int64_t)raw < p.extent;
            c2[i] = ok ? (lp & ((1 << p.page_shift) - 1)) * kPage : 0;
            c3[i] = ok ? raw : 0;
          } else {
            ok = (int64_t)lp * kPage < p.extent;
            c2[i] = ok ? lp * kPage : 0;
            c3[i] = it.b;
          }
          if (i < npg && !ok && lane == 0 && pw == 0) report(p.err, PA_DEVERR_PAGE_OOB, it.b, lp);
        }
        // box b = page (b % 8), 64-column slab (b / 8); this warp issues the
        // boxes b = sub + 2 * lane of its tensor
        const int my_box = sub + 2 * lane;
        const int my_page = my_box & (kTilePages - 1);
        const int my_slab = my_box / kTilePages;
        const bool issuer = my_slab < Tr::kHalves && my_page < npg;
        const int my_count = __popc(__ballot_sync(0xffffffffu, issuer));
        int mc2 = 0, mc3 = 0;
#pragma unroll
        for (int i = 0; i < kTilePages; ++i)
          if (i == my_page) {
            mc2 = c2[i];
            mc3 = c3[i];
          }
        if (lane == 0) {
          const bool ok =
              failed || (Tr::kSharedEmpty
                             ? (Tj < 2 || mbar_wait(&x_done[sbuf(Tj - 2)], sbuf_par(Tj - 2)))
                             : mbar_wait(&x_empty[s], par ^ 1));
          if (!ok) {
            report(p.err, PA_DEVERR_TIMEOUT, it.b, j);
            failed = true;
          }
          if (!failed) mbar_arrive_expect_tx(&x_full[s], (uint32_t)(my_count * 2048));
        }
        __syncwarp();
        // after a timeout this warp issues no further copy
        const bool stop = __shfl_sync(0xffffffffu, failed ? 1 : 0, 0) != 0;
        if (issuer && !stop)
          tma_load_4d(sX + s * Tr::kKVBytes + my_slab * Tr::kSlab + my_page * 2048, tm_x,
                      &x_full[s], my_slab * 64, g, mc2, mc3, pol_kv);
        __syncwarp();
        if (!stop) issued = Tj + 1;
      }
      tctr += it.ntiles;
      ++a;
    }
    // Copies in flight must land before the CTA exits, also when a consumer
    // stopped waiting after a timeout: wait (bounded) for the last stage
    // loads this warp issued and the last Q.  Each is the latest phase of its
    // barrier, so the parity test is exact.
    if (lane == 0) {
      for (int i = 1; i <= Tr::kStages && i <= issued; ++i) {
        const int tl = issued - i;
        mbar_wait(&x_full[tl % Tr::kStages], (uint32_t)((tl / Tr::kStages) & 1));
      }
      if (pw == 0 && q_issued >= 1) mbar_wait(q_full, (uint32_t)((q_issued - 1) & 1));
    }
    __syncwarp();
  } else if (warp == kWarpMMA || warp == kWarpQK) {
    // ======================= MMA issuers =======================
    // Warp 15 issues every S = Q K^T, warp 14 every O += P V, each from its
    // lane 0 and each committing its own instructions.  Split in two, each
    // issuer's chain of barrier round trips and commits per tile is half as
    // long, and the two chains overlap.  Q K^T of tile t writes the TMEM
    // buffer that holds P of tile t-3, so it waits for P V of that tile.
    bool failed = false;
    auto wait = [&](uint64_t* bar, uint32_t par, int where) {
      if (!failed && !mbar_wait(bar, par)) {
        report(p.err, PA_DEVERR_TIMEOUT, -1, where);
        failed = true;
      }
    };
    const bool bf = std::is_same<T, __nv_bfloat16>::value;
    const uint32_t id_qk = tc::idesc_f16(kBM, kBN, bf, false);
    const uint32_t id_pv = tc::idesc_f16(kBM, D, bf, true);
    // Descriptor bases, built once: a tile's operands sit at fixed offsets
    // from them, added to the start-address field (addr >> 4, 14 bits, never
    // carried out of the field since shared memory is below 256 KB).  The
    // issuing thread shares its scheduler with softmax warps, so every
    // instruction spent per MMA lengthens the tile.
    const uint64_t dQ = tc::smem_desc(smem_u32(sQ), 16, 1024);
    const uint64_t dK0 = tc::smem_desc(smem_u32(sK), 16, 1024);
    const uint64_t dV0 = tc::smem_desc(smem_u32(sV), Tr::kSlab, 1024);
    const bool is_qk = warp == kWarpQK;
    auto kv_par = [](int t) { return (uint32_t)((t / Tr::kStages) & 1); };
    int tctr = 0, a = 0;
    for (int wu = wu_first; wu < wu_end; wu = wu_next(wu)) {
      if (empty_half(sc, wu)) continue;
      const Item it = get_item<TB>(p, sc, wu >> 1, wu & 1);
      if (it.ntiles == 0) continue;
      if (is_qk) {
        wait(q_full, (uint32_t)(a & 1), 50);
        // Q into TMEM: Q K^T then reads only K from shared memory.  The copy
        // runs in order with this thread's MMAs (after the previous item's
        // last Q K^T, before this item's first), and frees Q's shared memory
        // for the next item once it has completed.
        tc::fence_after_sync();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tc::cp_128x256b(tQ + kk * 8, dQ + (((kk >> 2) * Tr::kSlab + (kk & 3) * 32) >> 4));
          tc::commit(q_empty);
        }
        __syncwarp();
        for (int j = 0; j < it.ntiles; ++j) {
          const int Tq = tctr + j;
          const int s = Tq % Tr::kStages;
          if (Tq >= kSBufs) {
            const uint32_t pd = sbuf_par(Tq - kSBufs);
            if (failed || !mbar_try_wait2(&k_full[s], kv_par(Tq), &pv_done[sbuf(Tq)], pd)) {
              wait(&k_full[s], kv_par(Tq), 100);
              wait(&pv_done[sbuf(Tq)], pd, 200);
            }
          } else {
            wait(&k_full[s], kv_par(Tq), 100);
          }
          tc::fence_after_sync();
          if (lane == 0) {
            const uint64_t dK = dK0 + (uint32_t)((s * Tr::kKVBytes) >> 4);
            const uint32_t tSq = tS(Tq);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = ((kk >> 2) * Tr::kSlab + (kk & 3) * 32) >> 4;
              tc::mma_f16_ts(tSq, tQ + kk * 8, dK + off, id_qk, kk > 0);
            }
            tc::commit(&s_full[sbuf(Tq)]);
            if (!Tr::kSharedEmpty) tc::commit(&k_empty[s]);
          }
          __syncwarp();
        }
      } else {
        for (int j = 0; j < it.ntiles; ++j) {
          const int Tj = tctr + j;
          const int s = Tj % Tr::kStages;
          {
            const uint32_t pp = sbuf_par(Tj);
            if (failed || !mbar_try_wait2(&p_full[sbuf(Tj)], pp, &v_full[s], kv_par(Tj))) {
              wait(&p_full[sbuf(Tj)], pp, 300);
              wait(&v_full[s], kv_par(Tj), 400);
            }
          }
          if (j == 0 && a >= 1) wait(o_free, (uint32_t)((a - 1) & 1), 450);
          // keys past the item's range: zero their V rows so P = 0 never meets a
          // stale or non-finite value
          const int valid = it.k1 - (it.k0 + j * kBN);
          if (valid < kBN) {
            uint8_t* vt = sV + s * Tr::kKVBytes;
            const int nrow = kBN - valid;
            for (int e = lane; e < nrow * Tr::kHalves * 8; e += 32) {
              const int r = valid + e / (Tr::kHalves * 8);
              const int rest = e % (Tr::kHalves * 8);
              *reinterpret_cast<uint4*>(vt + (rest >> 3) * Tr::kSlab + r * 128 + (rest & 7) * 16) =
                  make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          tc::fence_after_sync();
          if (lane == 0) {
            const uint64_t dV = dV0 + (uint32_t)((s * Tr::kKVBytes) >> 4);
            const uint32_t tP = tS(Tj);
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              tc::mma_f16_ts(tO, tP + kk * 8, dV + (kk * 2048 >> 4), id_pv,
                             (j > 0 || kk > 0) ? 1u : 0u);
            tc::commit(&pv_done[sbuf(Tj)]);
            if (!Tr::kSharedEmpty) tc::commit(&v_empty[s]);
          }
          __syncwarp();
        }
      }
      tctr += it.ntiles;
      ++a;
    }
    // every tcgen05 operation of both issuers has completed once both arrive
    if (lane == 0) tc::commit(mma_fin);
    __syncwarp();
    wait(mma_fin, 0, 900);
  } else if (warp < kSoftWarps) {
    // ======================= softmax warps 0-7 =======================
    // Warps w and w+4 own tile rows 32*(w%4) .. +31 (the TMEM lane quarter a
    // warp may access); warp w < 4 takes S columns 0-63 and O columns
    // [0, D/2), warp w >= 4 columns 64-127 and [D/2, D).  The two halves of a
    // row agree on the running max through shared memory and keep separate
    // partial sums, added at the end.
    const int quarter = warp & 3, hf = warp >> 2;
    const int r = quarter * 32 + lane;  // tile row == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float sc_l2 = p.scale_log2;
    float* xmax = reinterpret_cast<float*>(smem + Tr::kOffX);  // [2 parity][2 half][128]
    float* xl = xmax + 2 * 2 * 128;                             // [128]
    bool failed = false;
    auto wait = [&](uint64_t* bar, uint32_t par, int where) {
      if (!failed && !mbar_wait(bar, par)) {
        report(p.err, PA_DEVERR_TIMEOUT, -1, where);
        failed = true;
      }
    };
    auto pair_sync = [&]() { named_barrier(1 + quarter, 64); };
    constexpr int kDH = D / 2;  // O columns per half
    int tctr = 0, a = 0;
    for (int wu = wu_first; wu < wu_end; wu = wu_next(wu)) {
      if (empty_half(sc, wu)) continue;
      const Item it = get_item<TB>(p, sc, wu >> 1, wu & 1);
      const bool valid = r < it.nrows;
      const bool quarter_live = quarter * 32 < it.nrows;  // any valid row in this quarter
      int qi, h;
      if (it.kind == 0) {
        qi = it.qs + r;
        h = it.head;
      } else {
        qi = r / p.G;
        h = it.head * p.G + r % p.G;
      }
      int vis_end = p.causal ? min(it.k1, qi + it.lk - it.qlen + 1) : it.k1;
      if (!valid) vis_end = it.k0;
      const bool to_partial = it.kind == 1 && it.nsplit > 1;
      const int64_t grow = it.row0 + qi;
      const int64_t nrows_all = p.cu_seqlens_q ? (int64_t)p.total_q : (int64_t)p.B * p.Lq;
      auto write_half = [&](const float* ov, int c, float inv) {  // 32 columns at hf*kDH + c*32
        const int col = hf * kDH + c * 32;
        if (to_partial) {
          float* dst = p.o_part + (((int64_t)it.split * nrows_all + grow) * p.Hq + h) * D + col;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) =
                make_float4(ov[i] * inv, ov[i + 1] * inv, ov[i + 2] * inv, ov[i + 3] * inv);
        } else {
          T* dst = reinterpret_cast<T*>(p.out) + (grow * p.Hq + h) * D + col;
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 u;
            u.x = E::from_f2(ov[i] * inv, ov[i + 1] * inv);
            u.y = E::from_f2(ov[i + 2] * inv, ov[i + 3] * inv);
            u.z = E::from_f2(ov[i + 4] * inv, ov[i + 5] * inv);
            u.w = E::from_f2(ov[i + 6] * inv, ov[i + 7] * inv);
            *reinterpret_cast<uint4*>(dst + i) = u;
          }
        }
      };
      auto write_lse = [&](float v) {
        if (to_partial) {
          p.lse_part[((int64_t)it.split * nrows_all + grow) * p.Hq + h] = v;
        } else if (p.lse != nullptr) {
          if (p.cu_seqlens_q)
            p.lse[(int64_t)h * p.total_q + grow] = v;
          else
            p.lse[((int64_t)it.b * p.Hq + h) * p.Lq + qi] = v;
        }
      };
      if (it.ntiles == 0) {
        if (valid) {
          float z[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] = 0.f;
          for (int c = 0; c < kDH / 32; ++c) write_half(z, c, 0.f);
          if (hf == 0) write_lse(neg_inf());
        }
        continue;
      }
      float m_use = neg_inf(), l = 0.f;
      for (int j = 0; j < it.ntiles; ++j) {
        const int Tj = tctr + j;
        const uint32_t tSj = tS(Tj) + lane_off + hf * 64;
        wait(&s_full[sbuf(Tj)], sbuf_par(Tj), 500);
        tc::fence_after_sync();
        // keys [0, lim) of this half's 64 columns are visible to the row
        const int lim = vis_end - (it.k0 + j * kBN + hf * 64);
        const bool full = lim >= 64;
        float v[64];
        float mx = neg_inf();
        if (quarter_live) {
          tc::tmem_ld32(tSj, v);
          tc::tmem_ld32(tSj + 32, v + 32);
          tc::tmem_wait_ld();
          float mx8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) mx8[i] = neg_inf();
          if (full) {
#pragma unroll
            for (int i = 0; i < 64; ++i) mx8[i & 7] = fmaxf(mx8[i & 7], v[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 64; ++i) mx8[i & 7] = (i < lim) ? fmaxf(mx8[i & 7], v[i]) : mx8[i & 7];
          }
          mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                     fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
          if (mx != neg_inf()) mx *= sc_l2;
          xmax[((Tj & 1) * 2 + hf) * 128 + r] = mx;
        }
        tc::fence_before_sync();
        pair_sync();
        tc::fence_after_sync();  // the partner's S loads precede this half's P stores
        if (quarter_live) mx = fmaxf(mx, xmax[((Tj & 1) * 2 + (hf ^ 1)) * 128 + r]);
        // both halves of a row see the same maximum and decide alike
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
        // P (16-bit) goes into TMEM over this tile's S: the row's 64 keys of
        // this half -> columns [32 hf, 32 hf + 32) of the S buffer (both halves
        // of the row loaded their S before the exchange above).  P V of the
        // tile three back, which read the previous P there, completed before
        // the Q K^T that wrote this S was issued, so no wait is needed.
        if (quarter_live) {
          const float neg_m = -m_use;
          float rs8[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) rs8[i] = 0.f;
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {  // 16 columns (32 keys) per store
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int k = q2 * 32 + 2 * i;
              float e0 = ex2(fmaf(v[k], sc_l2, neg_m));
              float e1 = ex2(fmaf(v[k + 1], sc_l2, neg_m));
              if (!full) {
                e0 = (k < lim) ? e0 : 0.f;
                e1 = (k + 1 < lim) ? e1 : 0.f;
              }
              rs8[i & 7] += e0 + e1;
              pk[i] = E::from_f2(e0, e1);
            }
            tc::tmem_st16u(tS(Tj) + lane_off + hf * 32 + q2 * 16, pk);
          }
          l += ((rs8[0] + rs8[1]) + (rs8[2] + rs8[3])) + ((rs8[4] + rs8[5]) + (rs8[6] + rs8[7]));
        }
        if (j >= 1 && quarter_live && __any_sync(0xffffffffu, rescale)) {
          // O is stable once P V of the previous tile is done
          wait(&pv_done[sbuf(Tj - 1)], sbuf_par(Tj - 1), 650);
          tc::fence_after_sync();
          const float sa = rescale ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < kDH / 32; ++c) {
            float ov[32];
            const uint32_t ta = tO + lane_off + hf * kDH + c * 32;
            tc::tmem_ld32(ta, ov);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] *= sa;
            tc::tmem_st32(ta, ov);
          }
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&p_full[sbuf(Tj)]);
        }
      }
      // ---- epilogue: the two halves' sums, then O / l and LSE
      if (hf == 1) xl[r] = l;
      pair_sync();
      if (hf == 0) xl[r] = l + xl[r];
      pair_sync();
      const float L = xl[r];
      {
        const int tl = tctr + it.ntiles - 1;
        wait(&pv_done[sbuf(tl)], sbuf_par(tl), 700);
      }
      tc::fence_after_sync();
      const float inv = L > 0.f ? 1.f / L : 0.f;
      if (quarter_live) {
#pragma unroll 1
        for (int c = 0; c < kDH / 32; ++c) {
          float ov[32];
          tc::tmem_ld32(tO + lane_off + hf * kDH + c * 32, ov);
          tc::tmem_wait_ld();
          if (valid) write_half(ov, c, inv);
        }
        if (valid && hf == 0) write_lse(L > 0.f ? (m_use + lg2(L)) * kLn2 : neg_inf());
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(o_free);
      tctr += it.ntiles;
      ++a;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kWarpMMA) tc::tmem_dealloc(tbase, Tr::kTmemCols);
}

template <int D, typename T, bool TB>
cudaError_t launch_tb(const EngineParams& p, const CUtensorMap& q1, const CUtensorMap& q2,
                      const CUtensorMap& tk, const CUtensorMap& tv, int grid, cudaStream_t st) {
  using Tr = EngTraits<D>;
  static bool attr = false;
  if (!attr) {
    const cudaError_t e = cudaFuncSetAttribute(
        engine_kernel<D, T, TB>, cudaFuncAttributeMaxDynamicSharedMemorySize, Tr::kSmemBytes);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  engine_kernel<D, T, TB><<<grid, kThreads, Tr::kSmemBytes, st>>>(p, q1, q2, tk, tv);
  return cudaGetLastError();
}

template <int D, typename T>
cudaError_t launch_t(const EngineParams& p, const CUtensorMap& q1, const CUtensorMap& q2,
                     const CUtensorMap& tk, const CUtensorMap& tv, int grid, cudaStream_t st) {
  return p.tilebal ? launch_tb<D, T, true>(p, q1, q2, tk, tv, grid, st)
                   : launch_tb<D, T, false>(p, q1, q2, tk, tv, grid, st);
}

}  // namespace

int engine_grid() { return num_sms(); }

cudaError_t launch_engine(const EngineParams& p, const CUtensorMap& tm_q1,
                          const CUtensorMap& tm_q2, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, int D, int dtype, int grid, cudaStream_t st) {
  if (grid < 1) grid = 1;
  if (D == 128 && dtype == PA_F16) return launch_t<128, __half>(p, tm_q1, tm_q2, tm_k, tm_v, grid, st);
  if (D == 128 && dtype == PA_BF16)
    return launch_t<128, __nv_bfloat16>(p, tm_q1, tm_q2, tm_k, tm_v, grid, st);
  if (D == 64 && dtype == PA_F16) return launch_t<64, __half>(p, tm_q1, tm_q2, tm_k, tm_v, grid, st);
  if (D == 64 && dtype == PA_BF16)
    return launch_t<64, __nv_bfloat16>(p, tm_q1, tm_q2, tm_k, tm_v, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
