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
// as a normalised partial + LSE; the CTA that finishes a stream's last split
// merges its partials into the final rows (see "split merge" below), so a
// call is one launch.
//
// New tokens of a kvcache call (k=/v= append) are patched into the staged page
// from k_new/v_new and written to their cache slots by the CTA whose split
// covers them, so no CTA ever reads a slot another CTA is writing.
#include <type_traits>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

// Query blocks of 3-16 rows per kv head (GQA decode, short multi-query
// decode) run a tensor-core consumer: one warp per 16-token page computes
// S^T = K Q^T and O^T += V^T P^T with warp-level m16n8k16 MMAs (the 16 keys
// of the page as M, up to 8 query rows per N tile, fp32 accumulators in
// registers), so each key costs about one MMA instead of a CUDA-core dot
// product per row.  K/V pages arrive as 128-byte-swizzled 64-column TMA
// boxes, which ldmatrix reads without bank conflicts.
template <int D, typename T, int RMAX>
struct DecodeTraits {
  static constexpr bool kMma = RMAX >= 8;
  static constexpr int kStagePages = 4;
  // CUDA-core consumers: warps w and w + 4 take keys [0, 8) and [8, 16) of
  // page w of every stage.  Tensor-core consumer: warps w and w + 4 take page
  // w of even and odd stages respectively.
  static constexpr int kKeyParts = 2;
  static constexpr int kPartKeys = kPage / kKeyParts;
  static constexpr int kConsumerWarps = kStagePages * kKeyParts;
  // producer warps: one, or (tensor-core consumer, whose 64-column boxes are
  // half the size) one for K and one for V -- TMA issue throughput is per
  // issuing warp
  static constexpr int kProducers = kMma ? 2 : 1;
  static constexpr int kTensorsPerProducer = 2 / kProducers;
  static constexpr int kThreads = (kConsumerWarps + kProducers) * 32;
  static constexpr int kHalves = D / 64;  // 64-column boxes per page (tensor-core consumer)
  static constexpr int kStages =
      kMma ? ((D == 128) ? (RMAX == 8 ? 5 : 4) : 8) : ((D == 128) ? 3 : 5);
  static constexpr int kMinBlocks = kMma ? 1 : 2;
  static constexpr int kPageElems = kPage * D;
  static constexpr int kPageBytes = kPageElems * 2;
  static constexpr int kQCh = D / 64;  // 16-byte chunks per lane per key in QK
  static constexpr int kPVE = D / 32;  // output columns per lane
  // shared memory layout (bytes)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kStages * kStagePages * kPageBytes;
  static constexpr int kOffMerge = kOffV + kStages * kStagePages * kPageBytes;
  // merge area.  CUDA-core consumer: warps 1-7 leave (O, m, l) per row for
  // warp 0.  Tensor-core consumer: every warp leaves O [row][D + 4] (the pad
  // spreads its fragment stores over the banks) and (m, l) per row; warp w
  // merges rows w, w + 8.
  static constexpr int kORow = D + 4;
  static constexpr int kWarpMergeF = RMAX * kORow + 2 * RMAX;
  static constexpr int kMergeFloats = kMma ? kConsumerWarps * kWarpMergeF
                                           : (kConsumerWarps - 1) * RMAX * (D + 2);
  // tensor-core consumer: per warp, P of its page as [row][16 keys] 16-bit
  static constexpr int kOffP = kOffMerge + kMergeFloats * 4;
  static constexpr int al16(int x) { return (x + 15) & ~15; }
  static constexpr int kOffPrefix = al16(kOffP + (kMma ? kConsumerWarps * RMAX * kPage * 2 : 0));
  // per-sequence keys and cached keys of the scheduled batch
  static constexpr int kOffLens = al16(kOffPrefix + (kDecodeMaxSchedB + 1) * 4);
  static constexpr int kOffInfo = al16(kOffLens + 2 * kDecodeMaxSchedB * 4);
  static constexpr int kOffBar = al16(kOffInfo + kStages * kStagePages * 12);
  static constexpr int kOffMisc = al16(kOffBar + 2 * kStages * 8);
  static constexpr int kOffQ = kOffMisc + 64;  // [stage][RMAX][D] query rows of an item
  static constexpr int kQRowBytes = D * 2;
  // + 1024: the dynamic shared memory base is aligned up to 1024 bytes (the
  // 128-byte swizzle pattern of the TMA boxes repeats every 1024 bytes)
  static constexpr int kSmemBytes = ((kOffQ + kStages * RMAX * kQRowBytes) + 127) / 128 * 128 + 1024;
  static_assert(kOffBar % 8 == 0, "mbarriers need 8-byte alignment");
  static_assert(kOffV % 1024 == 0 && kOffMerge % 16 == 0, "TMA destinations and merge rows");
};

struct SeqInfo {
  int qlen;      // query rows of this sequence (Lq)
  int64_t row0;  // row index of its first query row in [B * Lq]
  int lk;        // keys attended
  int old;       // keys already in the cache
};

__device__ __forceinline__ SeqInfo seq_info(const DecodeParams& p, int b, bool report_errors) {
  SeqInfo si;
  si.qlen = p.Lq;
  si.row0 = (int64_t)b * p.Lq;
  si.old = __ldg(p.cache_seqlens + b);
  si.lk = si.old + p.Lnew;
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

// ---------------------------------------------------------------- warp MMA
// ldmatrix: four (or two) 8x8 16-bit matrices, each row address supplied by
// one lane (lanes 8j..8j+7 for matrix j); .trans transposes each matrix.
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];"
               : "=r"(r[0]), "=r"(r[1])
               : "r"(addr));
}
// D += A B, m16n8k16, A row-major 16x16, B column-major 16x8, fp32 accumulate.
template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
  }
}
template <typename T> __device__ __forceinline__ uint16_t to_bits(float x);
template <> __device__ __forceinline__ uint16_t to_bits<__half>(float x) {
  return __half_as_ushort(__float2half_rn(x));
}
template <> __device__ __forceinline__ uint16_t to_bits<__nv_bfloat16>(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Element offset of (row t, 16-byte chunk c) in a staged page: row-major rows
// of D elements, or (kSwz) 64-column halves of 16 rows x 128 bytes with the
// 128-byte swizzle of the TMA boxes (chunk c % 8 of a row stored at chunk
// position (c % 8) ^ (t % 8)).
template <int D, bool kSwz>
__device__ __forceinline__ int page_elem(int t, int c) {
  if constexpr (kSwz)
    return (c >> 3) * (kPage * 64) + t * 64 + (((c & 7) ^ (t & 7)) << 3);
  else
    return t * D + c * 8;
}

// Rotary embedding (RoFormer rotation, tables from the caller) of feature d
// of a new token's row x at position pos: the pair (x1, x2) of d becomes
// (x1 c - x2 s, x1 s + x2 c), computed in fp32 (each product of two 16-bit
// values is exact there) and rounded once to the storage type, as the
// rotated value is stored (k) or attended (q).  Features at or past rot_dim
// and positions outside the table (`ok` false; reported by the caller) pass
// through.
template <typename T>
__device__ __forceinline__ float rope_elem(const DecodeParams& p, const T* x, int d, int pos,
                                           bool ok) {
  if (!ok || d >= p.rot_dim) return static_cast<float>(x[d]);
  const int half = p.rot_dim >> 1;
  int q, i1, i2;
  bool first;
  if (p.rot_interleaved) {
    q = d >> 1;
    i1 = 2 * q;
    i2 = i1 + 1;
    first = (d & 1) == 0;
  } else {
    first = d < half;
    q = first ? d : d - half;
    i1 = q;
    i2 = q + half;
  }
  const float x1 = static_cast<float>(x[i1]);
  const float x2 = static_cast<float>(x[i2]);
  const float c = static_cast<float>(__ldg(reinterpret_cast<const T*>(p.rot_cos) + (int64_t)pos * half + q));
  const float sn = static_cast<float>(__ldg(reinterpret_cast<const T*>(p.rot_sin) + (int64_t)pos * half + q));
  const float y = first ? fmaf(x1, c, -(x2 * sn)) : fmaf(x1, sn, x2 * c);
  return static_cast<float>(Elem<T>::from_f(y));
}

// Whether position pos of sequence b is inside the rotary table; reports it
// (lane 0 of the caller's warp) when it is not.
__device__ __forceinline__ bool rope_pos_ok(const DecodeParams& p, int b, int pos, bool report_it) {
  const bool ok = pos >= 0 && pos < p.rot_len;
  if (!ok && report_it) report(p.err, PA_DEVERR_LENGTH, b, pos);
  return ok;
}

// New tokens of a kvcache call among keys [t0, t1) of a staged page: the
// staged copy is patched from k_new/v_new (k rotated at its position when the
// call has rotary embedding) and the tokens are written to their cache slots
// (each consumer warp patches only the keys it reads).
template <int D, typename T, bool kSwz>
__device__ __forceinline__ void patch_new_tokens(const DecodeParams& p, T* kp, T* vp,
                                                 const int* info, int b, int g, int t_base,
                                                 int old, int t0, int t1, int lane) {
  const int c2 = info[0], c3 = info[1];
  const bool ok = info[2] != 0;
  constexpr int kChunks = D / 8;  // 16-byte chunks per row
  for (int idx = lane; idx < (t1 - t0) * kChunks; idx += 32) {
    const int t = t0 + idx / kChunks;
    const int c = idx % kChunks;
    const int64_t src = (((int64_t)b * p.Lnew + (t_base + t - old)) * p.Hkv + g) * D + c * 8;
    uint4 kv = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.k_new) + src));
    const uint4 vv = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const T*>(p.v_new) + src));
    if (p.rot_cos != nullptr && c * 8 < p.rot_dim) {
      const int pos = t_base + t;
      const bool rok = rope_pos_ok(p, b, pos, true);
      const T* krow = reinterpret_cast<const T*>(p.k_new) + (src - c * 8);
      uint32_t w4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w4[e] = Elem<T>::from_f2(rope_elem<T>(p, krow, c * 8 + 2 * e, pos, rok),
                                 rope_elem<T>(p, krow, c * 8 + 2 * e + 1, pos, rok));
      kv = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    *reinterpret_cast<uint4*>(kp + page_elem<D, kSwz>(t, c)) = kv;
    *reinterpret_cast<uint4*>(vp + page_elem<D, kSwz>(t, c)) = vv;
    if (ok) {
      T* kdst = reinterpret_cast<T*>(p.k_cache) + (int64_t)c3 * p.k_sb + (int64_t)(c2 + t) * p.k_st +
                (int64_t)g * p.k_sh + c * 8;
      T* vdst = reinterpret_cast<T*>(p.v_cache) + (int64_t)c3 * p.v_sb + (int64_t)(c2 + t) * p.v_st +
                (int64_t)g * p.v_sh + c * 8;
      *reinterpret_cast<uint4*>(kdst) = kv;
      *reinterpret_cast<uint4*>(vdst) = vv;
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// ---------------------------------------------------------------- split merge
// The splits of a stream (one sequence, one kv head) are merged by the CTA
// that finishes last, inside this launch: no combine kernel and no state
// that has to start at zero.  Each stream has a 64-bit arrival word in the
// workspace holding (launch tag, count).  The launch tag is %gridid, a per-
// context launch number that every CTA of a grid reads alike, so a word
// holding arbitrary bytes or left by another launch counts as zero
// arrivals.  Replays of one CUDA graph may share a tag, so the arrival that
// completes a stream also resets its word to (tag, 0): every completed call
// leaves the words it used at zero arrivals for a replay.  The 48 low bits
// of %gridid are the tag; 16 bits count up to the split count.  No CTA
// waits on another: an arrival's compare-and-swap loop repeats only when
// another arrival changed the word, so it ends after at most as many rounds
// as there are splits.
__device__ __forceinline__ unsigned long long launch_tag() {
  unsigned long long id;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(id));
  return id & 0xffffffffffffull;
}

// One arrival on `word` for this launch; true for the arrival that makes
// `nb` of them, which leaves the word at (tag, 0).  The common case is one
// atomic add: a word that already carries this launch's tag counts the
// arrival.  An add that finds another tag (the first arrival after another
// launch, or bytes never written) went to a stale value; that arrival then
// installs (tag, 1) by compare-and-swap, unless another arrival of this
// launch has installed the tag meanwhile, in which case it adds itself to
// the installed count.  Every arrival is counted exactly once: by the one
// successful installation or by an add to a tagged word.
__device__ __forceinline__ bool arrive_last(unsigned long long* word, unsigned long long tag,
                                            int nb) {
  const unsigned long long mine = tag << 16;
  const unsigned long long old = atomicAdd(word, 1ull);
  unsigned long long cnt;
  if ((old >> 16) == tag) {
    cnt = (old & 0xffffull) + 1ull;
  } else {
    unsigned long long cur = old + 1ull;
    for (;;) {
      const unsigned long long prev = atomicCAS(word, cur, mine | 1ull);
      if (prev == cur) {
        cnt = 1ull;
        break;
      }
      if ((prev >> 16) == tag) {
        cnt = (atomicAdd(word, 1ull) & 0xffffull) + 1ull;
        break;
      }
      cur = prev;
    }
  }
  if (cnt < (unsigned long long)nb) return false;
  atomicExch(word, mine);
  return true;
}

// One warp merges the nb split partials of (row, h): O = sum_s w_s O_s / L,
// w_s = 2^(LSE_s log2 e - M), LSE = (M + log2 L) ln 2.  An empty split
// (LSE -inf) has weight 0.  The partial rows of the first kPre splits are
// loaded together with the LSEs (they lie in the workspace for every split
// index below s_max), so a merge of up to kPre splits waits on one round
// trip to memory rather than two.
template <int D, typename T>
__device__ __noinline__ void merge_split_row(const DecodeParams& p, int64_t row, int h, int qi,
                                             int b, int nb, int64_t nrows_all, int lane) {
  constexpr int kPVE = D / 32;
  constexpr int kPre = 4;
  const int64_t base = row * p.Hq + h;
  const int64_t sstride = nrows_all * p.Hq;
  float pre[kPre][kPVE];
#pragma unroll
  for (int j = 0; j < kPre; ++j) {
    if (j < nb) {
      const float* op = p.o_part + (j * sstride + base) * D + lane * kPVE;
      if constexpr (kPVE == 4) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(op));
        pre[j][0] = x.x;
        pre[j][1] = x.y;
        pre[j][2] = x.z;
        pre[j][3] = x.w;
      } else {
        const float2 x = __ldcg(reinterpret_cast<const float2*>(op));
        pre[j][0] = x.x;
        pre[j][1] = x.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < kPVE; ++e) pre[j][e] = 0.f;
    }
  }
  float M = neg_inf();
  float my_ls = neg_inf();
  for (int s = lane; s < nb; s += 32) {
    const float ls = __ldcg(p.lse_part + s * sstride + base) * kLog2e;
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
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      const float ls = __shfl_sync(0xffffffffu, my_ls, j);
      if (j < nb && ls != neg_inf()) {
        const float w = ex2(ls - M);
        L += w;
#pragma unroll
        for (int e = 0; e < kPVE; ++e) acc[e] = fmaf(w, pre[j][e], acc[e]);
      }
    }
    for (int s = kPre; s < nb; ++s) {
      const float ls = s < 32 ? __shfl_sync(0xffffffffu, my_ls, s)
                              : __ldcg(p.lse_part + s * sstride + base) * kLog2e;
      if (ls == neg_inf()) continue;
      const float w = ex2(ls - M);
      L += w;
      const float* op = p.o_part + (s * sstride + base) * D + lane * kPVE;
      if constexpr (kPVE == 4) {
        const float4 x = __ldcg(reinterpret_cast<const float4*>(op));
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
        acc[2] = fmaf(w, x.z, acc[2]);
        acc[3] = fmaf(w, x.w, acc[3]);
      } else {
        const float2 x = __ldcg(reinterpret_cast<const float2*>(op));
        acc[0] = fmaf(w, x.x, acc[0]);
        acc[1] = fmaf(w, x.y, acc[1]);
      }
    }
  }
  using E = Elem<T>;
  const float inv = L > 0.f ? 1.f / L : 0.f;
  T* orow = reinterpret_cast<T*>(p.out) + base * D + lane * kPVE;
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
    p.lse[((int64_t)b * p.Hq + h) * p.Lq + qi] = lse_v;
  }
}

// Called by all consumer warps of a CTA once each has written its partial
// rows of split `s` of stream (b, g): the arrival, and the merge if this
// split is the last of the stream's nb to finish.  Consumer warp w merges
// rows w, w + nwarps, ... of the R rows.
template <int D, typename T>
__device__ __forceinline__ void finish_split(const DecodeParams& p, int* sflag, int nwarps, int R,
                                             int b, int g, int nb, int64_t row0, int warp,
                                             int lane) {
  __threadfence();  // this thread's partial rows before the arrival
  named_barrier(1, nwarps * 32);
  if (warp == 0 && lane == 0)
    *sflag = arrive_last(p.split_ctr + (int64_t)b * p.Hkv + g, launch_tag(), nb) ? 1 : 0;
  named_barrier(1, nwarps * 32);
  if (*sflag == 0) return;
  __threadfence();  // every split's partial rows are visible past the last arrival
  const int64_t nrows_all = (int64_t)p.B * p.Lq;
  for (int r = warp; r < R; r += nwarps) {
    const int qi = r / p.G;
    merge_split_row<D, T>(p, row0 + qi, g * p.G + (r % p.G), qi, b, nb, nrows_all, lane);
  }
}

// Tensor-core consumer for 3-16 query rows per kv head (see DecodeTraits).
// Warp w owns page w % 4 of the stages whose sequence number has parity
// w / 4; every warp still waits for every stage and releases it (the item's
// query rows travel with its first stage).  Per page:
//   S^T[16 keys][8 rows] = K[16][D] Q^T[D][8]   D/16 MMAs per row tile, K by
//                                               ldmatrix, Q^T held in registers
//   online softmax per row (log2 domain); a lane holds keys k0 and k0 + 8 of
//   rows n0 and n0 + 1 of every row tile, the row max is shared by shuffles
//   P (16-bit) -> shared [row][16 keys] -> ldmatrix as the B operand
//   O^T[D][8 rows] += V^T[D][16] P^T[16][8]     D/16 MMAs per row tile, V^T by
//                                               ldmatrix.trans
// The eight warps' (m, l, O) are merged at the end of the item.
template <int D, typename T, int RMAX, typename NextWork, typename Pos>
__device__ __forceinline__ void mma_consume(const DecodeParams& p, uint8_t* smem,
                                            NextWork& next_work, Pos work0, int warp, int lane) {
  using Tr = DecodeTraits<D, T, RMAX>;
  using E = Elem<T>;
  constexpr int NT = RMAX / 8;  // row tiles (MMA N = 8 rows each)
  constexpr int KS = D / 16;    // QK^T k-steps; PV m-tiles of 16 columns
  T* sK = reinterpret_cast<T*>(smem + Tr::kOffK);
  T* sV = reinterpret_cast<T*>(smem + Tr::kOffV);
  float* sMerge = reinterpret_cast<float*>(smem + Tr::kOffMerge);
  uint16_t* sPw = reinterpret_cast<uint16_t*>(smem + Tr::kOffP) + warp * RMAX * kPage;
  const int* sInfo = reinterpret_cast<const int*>(smem + Tr::kOffInfo);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Tr::kOffBar);
  uint64_t* empty = full + Tr::kStages;
  const T* sQ = reinterpret_cast<const T*>(smem + Tr::kOffQ);
  int* sFlag = reinterpret_cast<int*>(smem + Tr::kOffMisc) + 1;

  const int k0 = lane >> 2;        // key of accumulator elements 0, 1 (k0 + 8: 2, 3)
  const int n0 = (lane & 3) * 2;   // rows n0, n0 + 1 of each row tile
  // ldmatrix row addresses: K as A (keys x features), V^T as A (features x
  // keys, transposed on load), P as B (rows x keys)
  const int qk_key = (lane & 7) + (((lane >> 3) & 1) << 3), qk_ch = lane >> 4;
  const int pv_key = (lane & 7) + ((lane >> 4) << 3), pv_ch = (lane >> 3) & 1;
  const uint32_t p_addr = smem_u32(sPw + (lane & 7) * kPage + ((lane >> 3) & 1) * 8);
  const float sl2 = p.scale_log2;
  const int wslot = warp % Tr::kStagePages;  // page of a stage this warp reads
  const uint32_t wpar = (uint32_t)(warp / Tr::kStagePages);  // parity of its stages

  uint32_t qctr = 0;  // stages of earlier items: ring position of this item's first stage
  bool failed = false;
  Pos wp = work0;
  int b, g, s, nb, p0, p1;
  SeqInfo si;
  while (next_work(wp, b, g, s, nb, p0, p1, si)) {
    const int R = si.qlen * p.G;  // <= RMAX for every item that exists
    const int kend = min(p1 * kPage, si.lk);
    int lim[NT][2];  // last key position rows n0, n0 + 1 of each tile may attend (-1: none)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int n = nt * 8 + n0 + j;
        lim[nt][j] = n < R ? (p.causal ? n / p.G + si.lk - si.qlen : 0x7fffffff) : -1;
      }
    uint32_t qb[NT][KS][2];
    float oacc[KS][NT][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[mt][nt][e] = 0.f;
    float m[NT][2], l[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = neg_inf();
      l[nt][0] = l[nt][1] = 0.f;
    }

    const int nstages = (p1 - p0 + Tr::kStagePages - 1) / Tr::kStagePages;
    for (int i = 0; i < nstages; ++i) {
      const uint32_t q = qctr + (uint32_t)i;
      const int stage = (int)(q % Tr::kStages);
      const uint32_t phase = (q / Tr::kStages) & 1u;
      const int pg = p0 + i * Tr::kStagePages;
      if (!failed && !mbar_wait(&full[stage], phase)) {
        report(p.err, PA_DEVERR_TIMEOUT, b, pg);
        failed = true;
      }
      if (i == 0) {
        // Q^T as the B operand: row k0 of each tile, features 16 kk + n0, +1
        // and + 8, + 9; rows past R are zero
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int row = nt * 8 + k0;
          const T* qrow = sQ + (stage * RMAX + row) * D + n0;
#pragma unroll
          for (int kk = 0; kk < KS; ++kk) {
            qb[nt][kk][0] = row < R ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk) : 0u;
            qb[nt][kk][1] = row < R ? *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8) : 0u;
          }
        }
      }
      const int page = pg + wslot;
      if ((q & 1u) == wpar && page < p1) {
        T* kp = sK + (stage * Tr::kStagePages + wslot) * Tr::kPageElems;
        T* vp = sV + (stage * Tr::kStagePages + wslot) * Tr::kPageElems;
        const int t_base = page * kPage;
        const int nvalid = min(kPage, kend - t_base);
        if (p.Lnew > 0 && t_base + nvalid > si.old)
          patch_new_tokens<D, T, true>(p, kp, vp, sInfo + (stage * Tr::kStagePages + wslot) * 3, b,
                                       g, t_base, si.old, max(si.old - t_base, 0), nvalid, lane);
        if (nvalid < kPage) {
          // rows past the keys get P = 0; zero their V so that no stale or
          // non-finite value meets it in the MMA
          for (int idx = lane; idx < (kPage - nvalid) * (D / 8); idx += 32) {
            const int t = nvalid + idx / (D / 8);
            *reinterpret_cast<uint4*>(vp + page_elem<D, true>(t, idx % (D / 8))) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          __syncwarp();
        }
        // ---- S^T = K Q^T
        float sacc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) sacc[nt][e] = 0.f;
        const uint32_t kbase = smem_u32(kp);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int c = 2 * kk + qk_ch;
          uint32_t a[4];
          ldsm_x4(a, kbase + (uint32_t)(page_elem<D, true>(qk_key, c) * 2));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816<T>(sacc[nt], a, qb[nt][kk]);
        }
        // ---- online softmax (log2 domain) and P to shared memory
        float al[NT][2];
        bool resc = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float x0 = (k0 < nvalid && t_base + k0 <= lim[nt][j]) ? sacc[nt][j] : neg_inf();
            const float x1 =
                (k0 + 8 < nvalid && t_base + k0 + 8 <= lim[nt][j]) ? sacc[nt][2 + j] : neg_inf();
            float mx = fmaxf(x0, x1);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const float mnew = fmaxf(m[nt][j], mx == neg_inf() ? mx : mx * sl2);
            float alpha = 1.f, e0 = 0.f, e1 = 0.f;
            if (mnew != neg_inf()) {
              alpha = ex2(m[nt][j] - mnew);
              e0 = ex2(fmaf(x0, sl2, -mnew));
              e1 = ex2(fmaf(x1, sl2, -mnew));
            }
            l[nt][j] = l[nt][j] * alpha + (e0 + e1);
            m[nt][j] = mnew;
            al[nt][j] = alpha;
            resc |= alpha != 1.f;
            uint16_t* prow = sPw + (nt * 8 + n0 + j) * kPage;
            prow[k0] = to_bits<T>(e0);
            prow[k0 + 8] = to_bits<T>(e1);
          }
        }
        if (__any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int mt = 0; mt < KS; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              oacc[mt][nt][0] *= al[nt][0];
              oacc[mt][nt][1] *= al[nt][1];
              oacc[mt][nt][2] *= al[nt][0];
              oacc[mt][nt][3] *= al[nt][1];
            }
        }
        __syncwarp();
        // ---- O^T += V^T P^T
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) ldsm_x2(pb[nt], p_addr + (uint32_t)(nt * 8 * kPage * 2));
        const uint32_t vbase = smem_u32(vp);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t a[4];
          ldsm_x4_t(a, vbase + (uint32_t)(page_elem<D, true>(pv_key, 2 * mt + pv_ch) * 2));
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma16816<T>(oacc[mt][nt], a, pb[nt]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }
    qctr += (uint32_t)nstages;

    // ---- merge the eight warps' softmax states: every warp leaves O [row][d]
    // and (m, l) per row; warp w then merges rows w and w + 8
    float* mw = sMerge + warp * Tr::kWarpMergeF;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float lj = l[nt][j];
        lj += __shfl_xor_sync(0xffffffffu, lj, 4);
        lj += __shfl_xor_sync(0xffffffffu, lj, 8);
        lj += __shfl_xor_sync(0xffffffffu, lj, 16);
        const int n = nt * 8 + n0 + j;
        if (k0 == 0) {
          mw[RMAX * Tr::kORow + 2 * n] = m[nt][j];
          mw[RMAX * Tr::kORow + 2 * n + 1] = lj;
        }
      }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int n = nt * 8 + n0 + (e & 1);
          const int d = 16 * mt + k0 + ((e >> 1) << 3);
          mw[n * Tr::kORow + d] = oacc[mt][nt][e];
        }
    named_barrier(1, Tr::kConsumerWarps * 32);
    const bool to_partial = nb > 1;
    const int64_t nrows_all = (int64_t)p.B * p.Lq;
    for (int r = warp; r < R; r += Tr::kConsumerWarps) {
      float M = neg_inf();
#pragma unroll
      for (int w = 0; w < Tr::kConsumerWarps; ++w)
        M = fmaxf(M, sMerge[w * Tr::kWarpMergeF + RMAX * Tr::kORow + 2 * r]);
      float Ls = 0.f;
      float acc[Tr::kPVE];
#pragma unroll
      for (int e = 0; e < Tr::kPVE; ++e) acc[e] = 0.f;
      if (M != neg_inf()) {
#pragma unroll
        for (int w = 0; w < Tr::kConsumerWarps; ++w) {
          const float* src = sMerge + w * Tr::kWarpMergeF;
          const float aw = ex2(src[RMAX * Tr::kORow + 2 * r] - M);
          Ls += src[RMAX * Tr::kORow + 2 * r + 1] * aw;
          const float* orow = src + r * Tr::kORow + lane * Tr::kPVE;
#pragma unroll
          for (int e = 0; e < Tr::kPVE; ++e) acc[e] = fmaf(orow[e], aw, acc[e]);
        }
      }
      const float inv = (Ls > 0.f) ? 1.f / Ls : 0.f;
      const float lse_v = (Ls > 0.f) ? (M + lg2(Ls)) * kLn2 : neg_inf();
      const int qi = r / p.G;
      const int h = g * p.G + (r % p.G);
      const int64_t row = si.row0 + qi;
      if (to_partial) {
        float* op = p.o_part + (((int64_t)s * nrows_all + row) * p.Hq + h) * D + lane * Tr::kPVE;
#pragma unroll
        for (int e = 0; e < Tr::kPVE; ++e) op[e] = acc[e] * inv;
        if (lane == 0) p.lse_part[((int64_t)s * nrows_all + row) * p.Hq + h] = lse_v;
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
        if (p.lse != nullptr && lane == 0) p.lse[((int64_t)b * p.Hq + h) * p.Lq + qi] = lse_v;
      }
    }
    if (to_partial)
      finish_split<D, T>(p, sFlag, Tr::kConsumerWarps, R, b, g, nb, si.row0, warp, lane);
    named_barrier(1, Tr::kConsumerWarps * 32);
  }
}

// Position of a CTA in its work: the next item index (direct, uniform) or
// the next page of its share of the concatenated streams (balanced).
struct WorkPos {
  int item;
  int x, x_end;
};

// Last index i in [0, n) with pre[i] <= x (pre non-decreasing, pre[0] <= x).
__device__ __forceinline__ int last_le_int(const int* pre, int n, int x) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

template <int D, typename T, int RMAX>
__global__ void __launch_bounds__(DecodeTraits<D, T, RMAX>::kThreads,
                                  DecodeTraits<D, T, RMAX>::kMinBlocks)
    decode_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                  const __grid_constant__ CUtensorMap tmv) {
  using Tr = DecodeTraits<D, T, RMAX>;
  using E = Elem<T>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  T* sK = reinterpret_cast<T*>(smem + Tr::kOffK);
  T* sV = reinterpret_cast<T*>(smem + Tr::kOffV);
  float* sMerge = reinterpret_cast<float*>(smem + Tr::kOffMerge);
  int* sPrefix = reinterpret_cast<int*>(smem + Tr::kOffPrefix);
  int* sLk = reinterpret_cast<int*>(smem + Tr::kOffLens);  // [B] keys (scheduled mode)
  int* sOld = sLk + kDecodeMaxSchedB;                        // [B] keys already cached
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
      mbar_init(&full[i], Tr::kProducers);
      mbar_init(&empty[i], Tr::kConsumerWarps);
    }
    fence_mbar_init();
  }
  if (warp == Tr::kConsumerWarps && lane == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }

  // ---- device work schedule, from the lengths on the GPU (no host read):
  //   direct    one split per sequence (kvcache call, s_max == 1): item i is
  //             (b, g) = (i / Hkv, i % Hkv), items dealt to the CTAs in turn.
  //   uniform   explicit num_splits: every sequence in min(pages, num_splits)
  //             splits of equal pages, items dealt in turn.
  //   balanced  automatic splits: the pages of all (sequence, kv head)
  //             streams, concatenated sequence by sequence, are cut into equal
  //             contiguous shares of `share` pages, one per CTA; the pieces a
  //             stream is cut into are its splits (consecutive CTAs).
  const bool direct = p.s_max <= 1;
  const bool balanced = !direct && p.target_ctas < kForcedSplitTarget && p.s_max >= 2;
  int num_items = 0;   // direct, uniform
  int chunk = 0;       // uniform: pages per split
  int share = 1;       // balanced: pages per CTA
  int total_pages = 0; // balanced: pages of all streams
  const SplitSched sch{p.s_max, p.target_ctas, p.min_chunk_pages};
  if (direct) {
    num_items = p.B * p.Hkv;
  } else {
    // Lengths of every sequence -> shared memory (item decoding reads them
    // there), pages -> sPrefix (scratch until the prefix sum replaces it),
    // and the longest sequence.
    int* sRed = reinterpret_cast<int*>(sMerge);
    int pmax = 0;
    for (int b = tid; b < p.B; b += Tr::kThreads) {
      const SeqInfo si = seq_info(p, b, true);
      const int pages = (si.lk + kPage - 1) / kPage;
      sPrefix[b] = pages;
      sLk[b] = si.lk;
      sOld[b] = si.old;
      pmax = max(pmax, pages);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pmax = max(pmax, __shfl_xor_sync(0xffffffffu, pmax, o));
    if (lane == 0) sRed[warp] = pmax;
    __syncthreads();
    pmax = 0;
    for (int w = 0; w < Tr::kThreads / 32; ++w) pmax = max(pmax, sRed[w]);
    if (!balanced) chunk = max(1, p.min_chunk_pages);
    __syncthreads();
    // prefix sums over the sequences (warp 0): uniform -> split counts,
    // balanced -> pages of all kv heads
    if (warp == 0) {
      int carry = 0;
      for (int base = 0; base < p.B; base += 32) {
        const int b = base + lane;
        int v = 0;
        if (b < p.B) {
          const int pages = sPrefix[b];
          if (balanced)
            v = pages * p.Hkv;
          else
            split_pages_per(sch, pages, chunk, &v);
        }
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (b < p.B) sPrefix[b] = carry + incl - v;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        sPrefix[p.B] = carry;
        sMisc[0] = carry;
      }
    }
    __syncthreads();
    if (!balanced) {
      num_items = sMisc[0] * p.Hkv;
    } else {
      total_pages = sMisc[0];
      // an equal share per CTA, at least min_chunk pages, and large enough
      // that no stream is cut into more than s_max pieces
      share = (total_pages + (int)gridDim.x - 1) / (int)gridDim.x;
      share = max(share, max(p.min_chunk_pages, (pmax + p.s_max - 2) / max(1, p.s_max - 1)));
      share = max(share, 1);
      // sequences without keys are in no share: their rows (O = 0, LSE =
      // -inf) are written here, by CTA b mod grid
      for (int b = blockIdx.x; b < p.B; b += gridDim.x) {
        if (sLk[b] != 0) continue;
        const int64_t row0 = (int64_t)b * p.Lq;
        const int nrow = p.Lq * p.Hq;
        for (int idx = tid; idx < nrow * (D / 8); idx += Tr::kThreads) {
          const int r = idx / (D / 8), c = idx % (D / 8);
          T* dst = reinterpret_cast<T*>(p.out) + (row0 + r / p.Hq) * p.Hq * D + (r % p.Hq) * D + c * 8;
          *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        if (p.lse != nullptr) {
          for (int r = tid; r < nrow; r += Tr::kThreads) {
            const int qi = r / p.Hq, h = r % p.Hq;
            p.lse[((int64_t)b * p.Hq + h) * p.Lq + qi] = neg_inf();
          }
        }
      }
    }
  }
  __syncthreads();

  // Work decoding shared by producer and consumers: lengths of a scheduled
  // sequence from shared memory (validated and reported by the prologue).
  auto seq_of = [&](int b, SeqInfo& si) {
    if (direct) {
      si = seq_info(p, b, true);
      return;
    }
    si.qlen = p.Lq;
    si.row0 = (int64_t)b * p.Lq;
    si.lk = sLk[b];
    si.old = sOld[b];
  };
  // The next work unit of this CTA: sequence b, kv head g, split s of nb,
  // pages [p0, p1).  Returns false when the CTA has none left.
  auto next_work = [&](WorkPos& w, int& b, int& g, int& s, int& nb, int& p0, int& p1,
                       SeqInfo& si) -> bool {
    if (!balanced) {
      if (w.item >= num_items) return false;
      g = w.item % p.Hkv;
      const int j = w.item / p.Hkv;
      w.item += gridDim.x;
      if (direct) {
        b = j;
        s = 0;
      } else {
        b = last_le_int(sPrefix, p.B, j);
        s = j - sPrefix[b];
      }
      seq_of(b, si);
      const int pages = (si.lk + kPage - 1) / kPage;
      const int per = direct ? pages : split_pages_per(sch, pages, chunk, &nb);
      if (direct) nb = 1;
      p0 = s * per;
      p1 = min(p0 + per, pages);
      if (p0 > p1) p0 = p1;
      return true;
    }
    if (w.x >= w.x_end) return false;
    b = last_le_int(sPrefix, p.B, w.x);
    seq_of(b, si);
    const int pages = (si.lk + kPage - 1) / kPage;  // > 0: w.x lies in this sequence's pages
    const int off = w.x - sPrefix[b];
    g = off / pages;
    p0 = off - g * pages;
    const int start = sPrefix[b] + g * pages;
    p1 = min(pages, p0 + (w.x_end - w.x));
    s = (int)blockIdx.x - start / share;
    nb = (start + pages - 1) / share - start / share + 1;
    w.x += p1 - p0;
    return true;
  };
  WorkPos work0;
  work0.item = blockIdx.x;
  work0.x = balanced ? min((int)blockIdx.x * share, total_pages) : 0;
  work0.x_end = balanced ? min(work0.x + share, total_pages) : 0;


  if (warp >= Tr::kConsumerWarps) {
    // ======================= producer warps =======================
    // The block-table entries of the item are read warp-wide, one page per
    // lane, 32 pages at a time and one batch ahead, so no stage waits on a
    // table load.  Each of the first lanes issues one K or V box of a stage's
    // pages.  Producer 0 loads K (and the query rows and the page records the
    // consumers' append patch reads) and producer 1 V; a single producer loads
    // both.
    const int pw = warp - Tr::kConsumerWarps;
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
    WorkPos wp = work0;
    int b, g, s, nb, p0, p1;
    SeqInfo si;
    while (next_work(wp, b, g, s, nb, p0, p1, si)) {
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
        // the box this lane issues: one full-row box per page and tensor
        // (CUDA-core consumers), or one per page, tensor and 64-column half
        // (tensor-core consumer); lanes [0, kBoxPerT) load K, the next V
        constexpr int kBoxPerT = Tr::kMma ? Tr::kStagePages * Tr::kHalves : Tr::kStagePages;
        const int w = Tr::kMma ? (lane % kBoxPerT) / Tr::kHalves : (lane & (Tr::kStagePages - 1));
        const int half = Tr::kMma ? lane % Tr::kHalves : 0;
        const int src = pg - base + w;
        const int c2 = __shfl_sync(0xffffffffu, cur2, src);
        const int c3 = __shfl_sync(0xffffffffu, cur3, src);
        const int ok = __shfl_sync(0xffffffffu, curok, src);
        if (pw == 0 && lane < kBoxPerT && half == 0 && w < n) {
          int* info = sInfo + (stage * Tr::kStagePages + w) * 3;
          info[0] = c2;
          info[1] = c3;
          info[2] = ok;
        }
        __syncwarp();
        // the item's query rows travel with its first stage: bulk-copied, or
        // with rotary embedding rotated by this warp, which then arrives
        // after writing them (the transaction bytes are announced first)
        const int nq = (pg == p0 && pw == 0) ? si.qlen * p.G : 0;
        const bool rot_q = nq > 0 && p.rot_cos != nullptr;
        if (lane == 0) {
          const uint32_t tx = (uint32_t)(n * Tr::kTensorsPerProducer * Tr::kPageBytes +
                                         (rot_q ? 0 : nq * Tr::kQRowBytes));
          if (rot_q)
            mbar_expect_tx(&full[stage], tx);
          else
            mbar_arrive_expect_tx(&full[stage], tx);
        }
        __syncwarp();
        if (!rot_q && lane < nq) {
          const int qi = lane / p.G;
          const int h = g * p.G + (lane % p.G);
          const T* qrow = reinterpret_cast<const T*>(p.q) + (int64_t)b * p.q_sb +
                          (int64_t)qi * p.q_st + (int64_t)h * p.q_sh;
          bulk_load(sQ + (stage * RMAX + lane) * D, qrow, Tr::kQRowBytes, &full[stage]);
        }
        if (lane < Tr::kTensorsPerProducer * kBoxPerT && w < n) {
          const bool is_k = Tr::kProducers == 1 ? lane < kBoxPerT : pw == 0;
          T* dst = (is_k ? sK : sV) + (stage * Tr::kStagePages + w) * Tr::kPageElems +
                   half * (kPage * 64);
          tma_load_4d(dst, is_k ? &tmk : &tmv, &full[stage], half * 64, g, c2, c3, pol);
        }
        if (rot_q) {
          // element e = r * D + d of the rows; four independent elements per
          // lane at a time, so that their loads overlap
          for (int e0 = 0; e0 < nq * D; e0 += 4 * 32) {
            float y[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int e = e0 + j * 32 + lane;
              const int r = e / D, d = e % D;
              y[j] = 0.f;
              if (e < nq * D) {
                const int qi = r / p.G;
                const int h = g * p.G + (r % p.G);
                const T* qrow = reinterpret_cast<const T*>(p.q) + (int64_t)b * p.q_sb +
                                (int64_t)qi * p.q_st + (int64_t)h * p.q_sh;
                // query row qi is the (Lnew - Lq + qi)-th new token
                const int pos = si.old + p.Lnew - si.qlen + qi;
                y[j] = rope_elem<T>(p, qrow, d, pos, rope_pos_ok(p, b, pos, d == 0));
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int e = e0 + j * 32 + lane;
              if (e < nq * D) sQ[(stage * RMAX + e / D) * D + e % D] = E::from_f(y[j]);
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&full[stage]);
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

  if constexpr (Tr::kMma) {
    mma_consume<D, T, RMAX>(p, smem, next_work, work0, warp, lane);
  } else {
    // ======================= consumers =======================
    int stage = 0;
    uint32_t phase = 0;
    bool failed = false;
    const int grp = lane >> 3;  // key slot within a QK pass
    const int sub = lane & 7;   // 16-byte chunk within the key row
    const int slot = warp % Tr::kStagePages;  // page of the stage this warp reads
    const int part = warp / Tr::kStagePages;  // which kPartKeys keys of that page

    WorkPos wp = work0;
    int b, g, s, nb, p0, p1;
    SeqInfo si;
    while (next_work(wp, b, g, s, nb, p0, p1, si)) {
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
          if (p.Lnew > 0 && t_base + min(nvalid, kb + Tr::kPartKeys) > si.old)
            patch_new_tokens<D, T, false>(p, kp, vp, sInfo + (stage * Tr::kStagePages + slot) * 3,
                                          b, g, t_base, si.old, max(si.old - t_base, kb),
                                          min(nvalid, kb + Tr::kPartKeys), lane);

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
      const bool to_partial = nb > 1;
      if (warp == 0) {
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
              float* op = p.o_part + (((int64_t)s * ((int64_t)p.B * p.Lq) + row) * p.Hq + h) * D;
  #pragma unroll
              for (int e = 0; e < Tr::kPVE; ++e) op[lane * Tr::kPVE + e] = acc[e] * inv;
              if (lane == 0)
                p.lse_part[((int64_t)s * ((int64_t)p.B * p.Lq) + row) * p.Hq + h] = lse_v;
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
              if (p.lse != nullptr && lane == 0) p.lse[((int64_t)b * p.Hq + h) * p.Lq + qi] = lse_v;
            }
          }
        }
      }
      if (to_partial)
        finish_split<D, T>(p, sMisc + 1, Tr::kConsumerWarps, R, b, g, nb, si.row0, warp, lane);
      named_barrier(1, Tr::kConsumerWarps * 32);
    }
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
  if (p.s_max <= 1)
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
    case 8: return launch_t<D, T, 8>(p, tmk, tmv, st);
    case 16: return launch_t<D, T, 16>(p, tmk, tmv, st);
  }
  return cudaErrorInvalidValue;
}

template <int D, typename T>
int occ_r(int rmax) {
  switch (rmax) {
    case 1: return occupancy_t<D, T, 1>();
    case 2: return occupancy_t<D, T, 2>();
    case 8: return occupancy_t<D, T, 8>();
    case 16: return occupancy_t<D, T, 16>();
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
