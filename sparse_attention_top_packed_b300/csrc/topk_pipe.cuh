// Warp-block kernel of the packed top-k + page transform (sm_103a).
//
// Operation (page "[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66% 끌어올린 Top-K 커널
// 최적화 분석", sglang PR #37889, Intro and sections 1-2): row i's window is
//   scores[i * row_stride + row_starts[i] + j], 0 <= j < seq_lens[i];
// the k largest are kept (a tie goes to the lower j), listed in ascending j and
// mapped through the row's page-table row; -1 pads windows shorter than k.
//
// Design (one CTA of 8 warps per row at a time, two CTAs per SM, rows strided
// over the persistent grid):
//
//  * Load.  A row's window, from its start rounded down to 16 bytes, is cut
//    into 128-byte units; warp w owns the w-th eighth of them, a contiguous
//    block, and streams it in 4 KB chunks (the last one partial) through its
//    own ring of kWStages shared-memory stages filled by 1-D TMA bulk copies
//    (L2 evict-first: every byte is read once).  Lane 0 refills a stage as
//    soon as the warp has taken it, so each warp keeps its next chunks -- also
//    those of its block of the next row -- in flight while a row is finished.
//    Lanes before the window start, past its end and past the block's end are
//    masked in registers (section 2 of the page, without writing the buffer).
//
//  * Admission.  Every row streams with a fixed threshold, a guess at a lower
//    bound of its k-th largest key: from the CTA's previous row (the key that
//    about 1.15 k of its candidates reach, scaled to the new length), or from
//    a strided sample of the row itself.  Each lane compares 32 consecutive
//    floats of a chunk with the threshold and appends the passing ones (order-
//    preserving key, window index) to the warp's region of the candidate
//    buffer, at positions from a prefix of the lanes' counts.  A region
//    therefore holds its candidates in ascending window index, and the regions
//    follow each other in warp order.  Each candidate is also counted in a
//    fine histogram: 2047 equal key bins above the threshold, sized so that
//    the k-th largest key lands in about bin 384.
//
//  * Selection.  The bin of the k-th largest key comes from the fine
//    histogram (each warp scans its 256 bins and publishes the scan; after one
//    barrier any warp finds a rank's bin alone).  Each warp compacts its region
//    in place to the entries at or above that bin, and the bin's own entries
//    (at most 32) are gathered and ranked by (key, ~j) in every warp, which
//    gives the exact k-th largest pair -- a tie goes to the lower j.  A bin of
//    more than 32 entries is settled by window order when they share one key,
//    else by a second fine level over the bin (2^11 sub-bins).  When the
//    histograms cannot settle it (the rank lies above their range, or the
//    sub-bin is still crowded with several keys), a radix select over the
//    buffer does.
//
//  * Emission.  Selected entries' output positions are prefix counts over the
//    ordered regions: each warp writes its selected window indices in
//    ascending order with ballots, no sorting.  The page transform of section
//    1 is applied in place while the next row streams (Deferred).
//
//  * Safety net.  If a threshold admitted fewer than k elements, or a region
//    overflowed, the row is streamed again from global memory in exact mode: a
//    threshold that starts at -inf and only ever rises to the k-th largest key
//    of the elements seen so far (so no selected element is dropped), a shared
//    buffer compacted when full, and a bitmap-ordered emission.
#pragma once

#include "topk_device.cuh"
#include "topk_sched.cuh"

#include <type_traits>

namespace topk {
namespace pipe {

constexpr int kThreads = 256;              // 8 warps
constexpr int kWarps = kThreads / 32;
constexpr int kBlock = kThreads;
constexpr int kWChunkQuads = 256;          // 4 KB: 8 consecutive quads (32 floats) per lane
constexpr int kWStages = 2;                // per-warp ring
constexpr int kChunkQuads = 1024;          // exact mode reads global memory 16 KB at a time
constexpr int kQuadsPerThread = kChunkQuads / kThreads;  // 4: quads tid + u * kThreads
constexpr int kHalfElems = kChunkQuads * 2;    // exact mode admits a chunk in two halves of 2048
constexpr int kKMax = 2048;
constexpr int kCap = 4096;                 // candidate buffer entries
constexpr int kRegion = kCap / kWarps;     // fast mode: one region of the buffer per warp
constexpr int kBins2 = 2048;               // refinement levels (<= 11 bits) / fine histogram
constexpr int kFineTop = kBins2 - 1;       // fine bins [0, kFineTop); keys above count apart
constexpr int kSegBits = kBins2 * 32;      // bitmap indices per emission segment
constexpr uint32_t kMaskBin = 0xFFE00000u;  // key bits of an exact-mode histogram bin (top 11)
constexpr uint32_t kMaskSub = 0xFFFFFC00u;  // key bits of a level-2 sub-bin

static_assert(kQuadsPerThread == 4, "exact mode: each thread takes four quads of a chunk");
// After an exact compaction the buffer holds k entries; a half chunk must fit.
static_assert(kCap - kKMax >= kHalfElems, "candidate buffer too small for k + half a chunk");
static_assert(kBins2 >= kKMax, "the output staging row reuses the level-2 histogram");
static_assert(kWChunkQuads == 8 * 32, "each lane takes 8 quads of a chunk");

// Admission / selection rule on the pair (key, nj = ~j): an element passes
// iff (key & mk, nj & mj) >= (tk, tj) lexicographically.  tf is a float with
// x >= tf <=> key(x) >= tk (tk has no bits outside mk), the fast first test.
struct Rule {
  uint32_t mk, tk, mj, tj;
  float tf;
  uint32_t exact;  // the pair test can reject an element that passed x >= tf
};

__device__ __forceinline__ Rule rule_prefix(uint32_t mk, uint32_t tk) {
  Rule a;
  a.mk = mk; a.tk = tk & mk; a.mj = 0u; a.tj = 0u;
  a.tf = key_floor_float(a.tk);
  a.exact = 0u;
  return a;
}

__device__ __forceinline__ Rule rule_all() { return rule_prefix(0u, 0u); }

__device__ __forceinline__ Rule rule_bin(uint32_t bin) { return rule_prefix(kMaskBin, bin << 21); }

__device__ __forceinline__ bool rule_pass(const Rule& a, uint32_t key, int32_t j) {
  const uint32_t kk = key & a.mk;
  return kk > a.tk || (kk == a.tk && ((~(uint32_t)j) & a.mj) >= a.tj);
}

// Lowest level-1 bin that can hold an admitted key under rule a.
__device__ __forceinline__ uint32_t rule_low_bin(const Rule& a) { return (a.mk & kMaskBin) ? a.tk >> 21 : 0u; }

struct PickOut {
  uint32_t bin, above, count;  // first target: bin holding rank r, count above it, its count
  uint32_t bin2, has2;         // second target (optional)
  uint32_t total;
};

// Per-warp TMA rings of NS stages of CQ quads for NW warps (one mbarrier per stage).
template <int NS, int NW = kWarps, int CQ = kWChunkQuads>
struct Ring {
  static constexpr int kChunk = CQ;
  float4 st[NW][NS][CQ];
  uint64_t full[NW][NS];
};

// Most streaming warps a kernel has (each fills its own part of the buffer).
constexpr int kMaxStreamWarps = 16;

// Shared state of one row in flight: candidate buffer, histogram, rules and
// the selection's scratch.
struct alignas(16) Shared {
  uint32_t bkey[kCap];
  int32_t bj[kCap];
  uint32_t hist2[kBins2];  // fine histogram / exact-mode histogram / refinement levels / bitmap
  uint32_t scratch[2][kWarps];
  uint32_t fsuf[kThreads];  // fine pick: bins of lanes >= this one in its warp's range
  uint32_t ftot[kWarps];    // fine pick: each warp's range of 256 bins
  PickOut pick[2];
  uint32_t wtot[kWarps];
  uint32_t rbase[kWarps], rcnt[kWarps];  // the buffer, as one region per warp
  uint32_t wmin[kWarps], wmax[kWarps], wtop[kWarps];
  uint32_t res_key[32];  // fast rows: the candidates of the fine bin holding rank k
  int32_t res_j[32];
  uint32_t res_w[32];    // and the warp whose region holds each
  uint32_t res_n;
  uint32_t scnt[kMaxStreamWarps];  // with more streaming warps than regions: each one's entry count
  uint32_t wcin[kWarps];            // fast rows: entries of the k-th key's bin in each warp's region
  uint32_t wkmin[kWarps], wkmax[kWarps];  // ... and their key range (crowded bins)
  uint32_t pad0_;
  uint32_t count;     // exact mode: entries in the shared buffer
  uint32_t overflow;  // fast mode: a region overflowed
  Rule rule;          // admission rule of the current row
  Rule hint;          // admission rule proposed for the next row
  uint32_t hint_valid;  // thread 0's: the next row may stream with S.hint
  uint32_t sample;      // this row takes its threshold from a sample (set with the row's rule)
  uint32_t hint_rank;  // rank the next row's hint should reach in this row (0: none)
  int32_t next_len;    // window length of the CTA's next row that needs a selection
  uint32_t fh_tk;      // fine histogram of this row: bins of 2^fh_sh keys from fh_tk
  uint32_t fh_sh;
  uint32_t hint_sh;    // fine shift proposed for the next row
};

struct Par {
  uint32_t p = 0, q = 0;
  __device__ __forceinline__ uint32_t* scratch(Shared& S) {
    uint32_t* s = S.scratch[p];
    p ^= 1u;
    return s;
  }
  __device__ __forceinline__ PickOut* slot(Shared& S) {
    PickOut* s = &S.pick[q];
    q ^= 1u;
    return s;
  }
};

// Barriers among the consumer warps only (named barrier 1).
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

__device__ __forceinline__ bool cbar_or(bool v) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\t"
               "setp.ne.u32 p, %1, 0;\n\t"
               "bar.red.or.pred q, 1, %2, p;\n\t"
               "selp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(r) : "r"(v ? 1u : 0u), "n"(kThreads) : "memory");
  return r != 0u;
}

// Exclusive prefix of v over the consumer threads; `total` gets the sum.
__device__ __forceinline__ uint32_t cta_excl_scan(uint32_t v, uint32_t* scratch, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan(v);
  if (lane == 31) scratch[warp] = incl;
  cbar();
  const uint32_t wt = lane < kWarps ? scratch[lane] : 0u;
  const uint32_t wincl = warp_incl_scan(wt);
  const uint32_t wexcl = __shfl_sync(0xFFFFFFFFu, wincl - wt, warp);
  total = __shfl_sync(0xFFFFFFFFu, wincl, kWarps - 1);
  return wexcl + incl - v;
}

// Block-wide bucket pick over NB bins (bins below `lo` count as empty): the
// bin where the count from the top first reaches r (and r2 when r2 > 0).
template <int NB>
__device__ __forceinline__ PickOut pick_bins(const uint32_t* hist, uint32_t lo, uint32_t r, uint32_t r2,
                                             Shared& S, Par& par) {
  constexpr int B = NB / kThreads;
  static_assert(B >= 1 && NB % kThreads == 0, "bins per thread");
  uint32_t* scratch = par.scratch(S);
  PickOut* slot = par.slot(S);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t h[B];
  if constexpr (B % 4 == 0) {
#pragma unroll
    for (int i = 0; i < B; i += 4) {
      const uint4 v = *reinterpret_cast<const uint4*>(hist + t * B + i);
      h[i] = v.x; h[i + 1] = v.y; h[i + 2] = v.z; h[i + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < B; ++i) h[i] = hist[t * B + i];
  }
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < B; ++i) {
    if ((uint32_t)(t * B + i) < lo) h[i] = 0u;
    s += h[i];
  }
  const uint32_t incl = warp_incl_suffix(s);
  if (lane == 0) scratch[warp] = incl;
  if (t == 0) *slot = PickOut{0u, 0u, 0u, 0u, 0u, 0u};
  cbar();
  const uint32_t wt = lane < kWarps ? scratch[lane] : 0u;
  const uint32_t wsuf = warp_incl_suffix(wt);
  const uint32_t above_warps = __shfl_sync(0xFFFFFFFFu, wsuf - wt, warp);
  const uint32_t total = __shfl_sync(0xFFFFFFFFu, wsuf, 0);
  uint32_t run = above_warps + incl - s;  // bins owned by higher threads
#pragma unroll
  for (int i = B - 1; i >= 0; --i) {
    const uint32_t prev = run;
    run += h[i];
    if (prev < r && run >= r) {
      slot->bin = (uint32_t)(t * B + i);
      slot->above = prev;
      slot->count = h[i];
    }
    if (r2 != 0u && prev < r2 && run >= r2) {
      slot->bin2 = (uint32_t)(t * B + i);
      slot->has2 = 1u;
    }
  }
  if (t == 0) slot->total = total;
  cbar();
  return *slot;
}

// Keeps the buffer entries i < n that pass `rule` (any order); returns the
// new count, also stored in S.count.  Starts and ends with a barrier.
__device__ __noinline__ uint32_t filter_buffer(Shared& S, uint32_t n, const Rule rule) {
  Par par;  // entered through a barrier: no thread still reads the scratch
  constexpr int E = kCap / kThreads;
  const int t = threadIdx.x;
  uint32_t key[E];
  int32_t jj[E];
  uint32_t keep = 0, c = 0;
  cbar();
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const uint32_t i = (uint32_t)(t * E + e);
    key[e] = 0u;
    jj[e] = 0;
    if (i < n) {
      key[e] = S.bkey[i];
      jj[e] = S.bj[i];
      if (rule_pass(rule, key[e], jj[e])) {
        keep |= 1u << e;
        ++c;
      }
    }
  }
  uint32_t total;
  uint32_t pos = cta_excl_scan(c, par.scratch(S), total);  // contains a barrier
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if (keep & (1u << e)) {
      S.bkey[pos] = key[e];
      S.bj[pos] = jj[e];
      ++pos;
    }
  }
  if (t == 0) S.count = total;
  cbar();
  return total;
}

// The buffer as kWarps regions, each scanned by one warp: entries
// [rbase[w], rbase[w] + rcnt[w]).  Each warp's lane 0 writes its own pair;
// a consumer barrier must follow before other warps read them.
__device__ __forceinline__ void set_regions_contiguous(Shared& S, uint32_t n) {
  const uint32_t per = (n + kWarps - 1) / kWarps, w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    const uint32_t b = min(w * per, n);
    S.rbase[w] = b;
    S.rcnt[w] = min(per, n - b);
  }
}

__device__ __forceinline__ uint64_t pair_of(uint32_t key, int32_t j) {
  return ((uint64_t)key << 32) | (uint64_t)(~(uint32_t)j);
}

__device__ __forceinline__ Rule rule_of_pair_prefix(uint64_t M, uint64_t T) {
  Rule a;
  a.mk = (uint32_t)(M >> 32);
  a.tk = (uint32_t)(T >> 32);
  a.mj = (uint32_t)M;
  a.tj = (uint32_t)T;
  a.tf = key_floor_float(a.tk);
  a.exact = a.mj != 0u ? 1u : 0u;
  return a;
}

// Exact rule that selects the r largest pairs (key, ~j) among the n buffered
// entries (r <= n; regions set).  The selected entries are those whose pair,
// under the returned prefix mask, is at least the returned prefix.
//
// With r2 > 0 it also proposes a key-prefix threshold that at least r2
// entries reach (the next row's hint): the deepest prefix, at most two digits
// below the common one, whose bin holds rank r2.  *hint_ok is 0 when fewer
// than r2 entries are buffered.
//
// `ready`: hist2 is all zero and S.wmin / S.wmax hold every region's key
// range (the fast stream leaves both so); otherwise they are made here.
struct Selection {
  Rule sel;   // selects the r largest pairs
  Rule hint;  // key-prefix rule reaching rank r2 (valid when hint_ok)
  uint32_t hint_ok;
};

__device__ __noinline__ Selection select_buffer(Shared& S, uint32_t n, uint32_t r, uint32_t r2, bool ready = false) {
  Par par;  // every pick below follows a barrier
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t base = S.rbase[w], cnt = S.rcnt[w];
  uint32_t mn = 0xFFFFFFFFu, mx = 0u;
  if (!ready) {
    // common prefix of the buffered keys
    for (uint32_t i = lane; i < cnt; i += 32) {
      const uint32_t key = S.bkey[base + i];
      mn = min(mn, key);
      mx = max(mx, key);
    }
    mn = __reduce_min_sync(0xFFFFFFFFu, mn);
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) {
      S.wmin[w] = mn;
      S.wmax[w] = mx;
    }
    cbar();
  }
#pragma unroll
  for (int i = 0; i < kWarps; ++i) {
    mn = min(mn, S.wmin[i]);
    mx = max(mx, S.wmax[i]);
  }
  const int P = mn == mx ? 32 : __clz(mn ^ mx);
  uint64_t M = P ? (~0ull << (64 - P)) : 0ull;
  uint64_t T = ((uint64_t)mn << 32) & M;
  int pos = 64 - P;
  uint32_t rem = r, hr = r2;
  bool track = r2 != 0u && r2 <= n;
  uint64_t HM = M, HT = T;
  for (int level = 0; pos > 0; ++level) {
    const int wd = pos < 11 ? pos : 11, sh = pos - wd;
    const uint32_t nb = 1u << wd;
    if (level > 0 || !ready) {
      for (uint32_t b = threadIdx.x; b < (uint32_t)kBins2; b += kThreads) S.hist2[b] = 0u;
      cbar();
    }
    for (uint32_t i = lane; i < cnt; i += 32) {
      const uint64_t c = pair_of(S.bkey[base + i], S.bj[base + i]);
      if ((c & M) == T) atomicAdd(&S.hist2[(uint32_t)(c >> sh) & (nb - 1u)], 1u);
    }
    cbar();
    const PickOut pk = pick_bins<kBins2>(S.hist2, 0u, rem, track ? hr : 0u, S, par);
    const uint64_t dm = (uint64_t)(nb - 1u) << sh;
    if (track && pk.has2) {
      HM = M | dm;
      HT = T | ((uint64_t)pk.bin2 << sh);
    }
    track = track && pk.has2 && pk.bin2 == pk.bin && level < 1;
    if (track) hr -= pk.above;
    M |= dm;
    T |= (uint64_t)pk.bin << sh;
    rem -= pk.above;
    pos = sh;
    if (pk.count == rem) break;
  }
  Selection out;
  out.sel = rule_of_pair_prefix(M, T);
  out.hint_ok = (r2 != 0u && r2 <= n) ? 1u : 0u;
  out.hint = rule_prefix((uint32_t)(HM >> 32), (uint32_t)(HT >> 32));  // the key part: never higher
  return out;
}

// The buffer would overflow: raise the threshold.  attempt 0 moves it to the
// level-1 bin of the k-th largest buffered key; attempt 1 (or when that does
// not rise) to the exact k-th largest pair.  n > k entries are buffered.
__device__ __noinline__ void compact(Shared& S, uint32_t n, uint32_t k, int attempt) {
  Par par;
  const Rule cur = S.rule;  // read before filter_buffer's first barrier; written after it
  const uint32_t lo = rule_low_bin(cur);
  if (attempt == 0 && !cur.exact) {
    cbar();
    const PickOut p1 = pick_bins<kBins2>(S.hist2, lo, k, 0u, S, par);
    if (p1.bin > lo || cur.mk == 0u) {
      const Rule a = rule_bin(p1.bin);
      filter_buffer(S, n, a);
      if (threadIdx.x == 0) S.rule = a;
      cbar();
      return;
    }
  }
  set_regions_contiguous(S, n);
  cbar();
  const Rule a = select_buffer(S, n, k, 0u).sel;
  const uint32_t kept = filter_buffer(S, n, a);
  // hist2 must count the buffer exactly again (the selection used it, and the
  // bin of the threshold lost entries)
  for (int b = threadIdx.x; b < kBins2; b += kThreads) S.hist2[b] = 0u;
  if (threadIdx.x == 0) S.rule = a;
  cbar();
  for (uint32_t i = threadIdx.x; i < kept; i += kThreads) atomicAdd(&S.hist2[S.bkey[i] >> 21], 1u);
  cbar();
}

// Exact mode reads a chunk from global memory as two halves of 8 elements a
// thread: with 32-bit elements a thread's quads 2h and 2h + 1 (kThreads
// apart), with 16-bit ones its quad h.  A chunk is exact_chunk_quads<E>()
// quads.
template <class E>
__device__ __forceinline__ constexpr int64_t exact_chunk_quads() {
  return (int64_t)kThreads * 2 * (8 / E::kPerQuad);
}

template <class E>
__device__ __forceinline__ void take_half(const Row& r, int64_t nq, int64_t cq, int h, float x[8]) {
  if constexpr (E::kPerQuad == 4) {
    float4 v[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t q = cq + threadIdx.x + (2 * h + u) * kThreads;
      v[u] = q < nq ? load_window_quad(r, q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    x[0] = v[0].x; x[1] = v[0].y; x[2] = v[0].z; x[3] = v[0].w;
    x[4] = v[1].x; x[5] = v[1].y; x[6] = v[1].z; x[7] = v[1].w;
  } else {
    const int64_t q = cq + threadIdx.x + h * kThreads;
    const float4 v = q < nq ? load_window_quad<E::kPerQuad>(r, q) : make_float4(0.f, 0.f, 0.f, 0.f);
    float y[8];
    E::decode(v, y);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = y[e];
  }
}

// Window index of the thread's element 0 of half h of the chunk at quad cq.
template <class E>
__device__ __forceinline__ int64_t half_first_index(const Row& r, int64_t cq, int h) {
  if constexpr (E::kPerQuad == 4) return (cq + threadIdx.x) * 4 - r.head + (int64_t)h * 8 * kThreads;
  return (cq + threadIdx.x + (int64_t)h * kThreads) * 8 - r.head;
}

// x[e] for a run-time e in [0, 8), as a tree of selects (indexing the array
// with a run-time value would move it to local memory).
__device__ __forceinline__ float pick8(const float x[8], int e) {
  const float a = (e & 1) ? x[1] : x[0], b = (e & 1) ? x[3] : x[2];
  const float c = (e & 1) ? x[5] : x[4], d = (e & 1) ? x[7] : x[6];
  const float lo = (e & 2) ? b : a, hi = (e & 2) ? d : c;
  return (e & 4) ? hi : lo;
}

// Window index of element e of a half whose element 0 has index jb0.  With
// 32-bit elements, elements 0-3 are one quad (index jb0 + e) and 4-7 the quad
// kThreads further on (index jb0 + 4 * kThreads + e - 4); with 16-bit ones
// the 8 elements are one quad.
template <class E>
__device__ __forceinline__ int32_t index8(int64_t jb0, int e) {
  if constexpr (E::kPerQuad == 4) return (int32_t)(jb0 + (e & 3) + ((e & 4) ? 4 * kThreads : 0));
  return (int32_t)(jb0 + e);
}

// Bit e set when element e of a half (laid out as index8) passes `rule` and
// lies in the window [0, L).
template <class E>
__device__ __forceinline__ uint32_t admit_mask(const Rule& rule, const float x[8], int64_t jb0, bool edge,
                                               int32_t L) {
  uint32_t m = 0u;
#pragma unroll
  for (int e = 0; e < 8; ++e) m |= (x[e] >= rule.tf ? 1u : 0u) << e;
  if (edge) {
    uint32_t valid = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int64_t j = index8<E>(jb0, e);
      valid |= (j >= 0 && j < L ? 1u : 0u) << e;
    }
    m &= valid;
  }
  if (rule.exact && m) {
    for (uint32_t mm = m; mm; mm &= mm - 1u) {
      const int e = __ffs(mm) - 1;
      if (!rule_pass(rule, key_of(pick8(x, e)), index8<E>(jb0, e))) m &= ~(1u << e);
    }
  }
  return m;
}

// Exact mode: appends the flagged elements of a half at pos, pos+1, ... and
// counts them in the histogram of the key's top 11 bits (hist2).
template <class E>
__device__ __forceinline__ void append(Shared& S, const float x[8], uint32_t m, uint32_t pos, int64_t jb0) {
  for (uint32_t mm = m; mm; mm &= mm - 1u) {
    const int e = __ffs(mm) - 1;
    const uint32_t key = key_of(pick8(x, e));
    if (in_bounds(pos < (uint32_t)kCap, kSiteCandidate)) {
      S.bkey[pos] = key;
      S.bj[pos] = index8<E>(jb0, e);
    }
    ++pos;
    atomicAdd(&S.hist2[key >> 21], 1u);
  }
}

// Exact mode: the row's window, straight from global memory, with a rising
// threshold starting at -inf; the buffer (one shared region, kCap entries) is
// compacted whenever a half chunk would overflow it.  One block-wide vote per
// half chunk.  For rows whose fast pass failed (rare).
template <class E = ElemF32>
__device__ __noinline__ void stream_row_exact(Shared& S, const Params& p, const Row r, int64_t nq) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint32_t k = (uint32_t)p.k;
  constexpr int64_t kCQ = exact_chunk_quads<E>();
  const int64_t nch = (nq + kCQ - 1) / kCQ;
  Rule rule = S.rule;
  for (int64_t c = 0; c < nch; ++c) {
    const int64_t cq = c * kCQ;
    const bool edge = c == 0 || c == nch - 1;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float xh[8];
      take_half<E>(r, nq, cq, h, xh);
      const int64_t jb0 = half_first_index<E>(r, cq, h);
      uint32_t m = admit_mask<E>(rule, xh, jb0, edge, r.L);
      uint32_t pos;
      for (int attempt = 0;; ++attempt) {
        const uint32_t n = __popc(m);
        const uint32_t incl = warp_incl_scan(n);
        const uint32_t wsum = __shfl_sync(0xFFFFFFFFu, incl, 31);
        uint32_t base = 0u;
        if (lane == 31) {
          if (wsum) base = atomicAdd(&S.count, wsum);
          S.wtot[w] = wsum;
        }
        base = __shfl_sync(0xFFFFFFFFu, base, 31);
        pos = base + incl - n;
        const bool ovf = cbar_or(wsum != 0u && base + wsum > (uint32_t)kCap);
        if (!ovf) break;
        // roll back this half chunk's reservations and raise the threshold
        uint32_t added = 0;
#pragma unroll
        for (int i = 0; i < kWarps; ++i) added += S.wtot[i];
        const uint32_t held = S.count - added;
        compact(S, held, k, attempt);
        rule = S.rule;
        for (uint32_t mm = m; mm; mm &= mm - 1u) {
          const int e = __ffs(mm) - 1;
          if (!rule_pass(rule, key_of(pick8(xh, e)), index8<E>(jb0, e))) m &= ~(1u << e);
        }
      }
      append<E>(S, xh, m, pos, jb0);
    }
  }
}

// Exact-mode rows (buffer in no particular order): writes the entries that
// pass `sel` (exactly k of them) in ascending window index, through the page
// transform, to out_row[0, k), ordering them with a bitmap of the window in
// hist2 (kSegBits indices per segment).
__device__ __noinline__ void emit_selected(Shared& S, const Params& p, const Row r, int64_t row, const Rule sel) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t rbase = S.rbase[warp], rcnt = S.rcnt[warp];
  uint32_t* bm = S.hist2;
  const uint32_t k = (uint32_t)p.k;
  int32_t* o = p.out + row * p.k;
  uint32_t out_base = 0;
  for (int64_t seg = 0; seg < r.L; seg += kSegBits) {
    const int32_t seg_lo = (int32_t)seg;
    const int32_t span = (int32_t)min((int64_t)kSegBits, (int64_t)r.L - seg);
    const int32_t nw = (span + 31) >> 5;
    cbar();  // previous users of the bitmap are done
    for (int i = 4 * t; i < nw; i += 4 * kThreads) *reinterpret_cast<uint4*>(bm + i) = make_uint4(0u, 0u, 0u, 0u);
    cbar();
    for (uint32_t i = lane; i < rcnt; i += 32) {
      const int32_t j = S.bj[rbase + i];
      if (j >= seg_lo && j - seg_lo < span && rule_pass(sel, S.bkey[rbase + i], j))
        atomicOr(&bm[(j - seg_lo) >> 5], 1u << ((j - seg_lo) & 31));
    }
    cbar();
    // warp w owns a run of whole 32-word rounds of the bitmap; in each round
    // lane l takes word round * 32 + l, so the ranks come from warp scans
    const int32_t wpw = ((nw + kWarps * 32 - 1) / (kWarps * 32)) * 32;
    const int32_t a0 = min(warp * wpw, nw), a1 = min(a0 + wpw, nw);
    uint32_t cnt = 0;
    for (int32_t i = a0 + lane; i < a1; i += 32) cnt += __popc(bm[i]);
    const uint32_t wsum = __reduce_add_sync(0xFFFFFFFFu, cnt);
    if (lane == 0) S.wtot[warp] = wsum;
    cbar();
    uint32_t pos0 = out_base, total = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) {
      const uint32_t v = S.wtot[i];
      pos0 += i < warp ? v : 0u;
      total += v;
    }
    for (int32_t i0 = a0; i0 < a1; i0 += 32) {
      const int32_t i = i0 + lane;
      const uint32_t word = i < a1 ? bm[i] : 0u;
      const uint32_t c = __popc(word);
      const uint32_t incl = warp_incl_scan(c);
      uint32_t pos = pos0 + incl - c;
      for (uint32_t b = word; b; b &= b - 1u) {
        if (pos < k)
          o[pos] = page_slot(r.page_row, p.page_bits, seg_lo + i * 32 + (__ffs(b) - 1), r.L);
        else
          atomicOr(&g_device_flags, kFlagBadOutputPosition);  // never expected
        ++pos;
      }
      pos0 += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    out_base += total;
  }
  cbar();  // every thread is done with the bitmap (hist2) and S.wtot
}

// ---------------------------------------------------------------------------
// Per-warp rings.
// ---------------------------------------------------------------------------

// Warp w's block of a row's aligned quads [0, nq): quads [q0, q1), contiguous,
// in warp order, cut at 128-byte units (8 quads) so that the blocks differ by
// at most one unit.  Its chunks are kWChunkQuads quads from q0 on, the last one
// partial.
template <int NB>
__device__ __forceinline__ void warp_block_of(int64_t nq, int w, int64_t& q0, int64_t& q1) {
  const int64_t nu = (nq + 7) >> 3;
  q0 = min(((nu * w) / NB) * 8, nq);
  q1 = min(((nu * (w + 1)) / NB) * 8, nq);
}

__device__ __forceinline__ void warp_block(int64_t nq, int w, int64_t& q0, int64_t& q1) {
  warp_block_of<kWarps>(nq, w, q0, q1);
}

// A row's descriptor as loaded; the Row is derived from it.
struct RowRaw {
  int32_t L, start, table_row;
};

__device__ __forceinline__ RowRaw load_row_raw(const Params& p, int64_t row) {
  RowRaw x = {0, 0, (int32_t)row};
  if (!row_index_ok(p, row)) return x;
  x.L = __ldg(p.seq_lens + row);
  x.start = __ldg(p.row_starts + row);
  x.table_row = p.row_to_batch ? __ldg(p.row_to_batch + row) : (int32_t)row;
  return x;
}

// Address of element `col` of buffer row `row` (elements of type E).
template <class E = ElemF32>
__device__ __forceinline__ uintptr_t elem_addr(const Params& p, int64_t row, int64_t col) {
  return reinterpret_cast<uintptr_t>(p.scores) + (uintptr_t)((row * p.row_stride + col) * E::kBytes);
}

// Quads of 16 bytes that hold the window of r (from its rounded-down start).
template <class E = ElemF32>
__device__ __forceinline__ int64_t quads_of(const Row& r) {
  return ((int64_t)r.L + r.head + E::kPerQuad - 1) / E::kPerQuad;
}

template <class E = ElemF32>
__device__ __forceinline__ Row make_row(const Params& p, int64_t row, const RowRaw& x) {
  check_row_window(p, x.L, x.start);
  Row r;
  r.L = x.L > 0 ? x.L : 0;
  const uintptr_t a = elem_addr<E>(p, row, x.start);
  r.head = (int32_t)((a & 15u) / E::kBytes);
  r.base4 = reinterpret_cast<const float4*>(a & ~(uintptr_t)15u);
  r.page_row = p.page_table ? p.page_table + (int64_t)x.table_row * p.pt_stride : nullptr;
  return r;
}

// A warp's cursor over its chunk sequence: the warp's block of each of the
// CTA's rows (its contiguous range [lo, hi), rows with seq_len > k).
// Uniform across the warp.
struct WCursor {
  const float4* src;
  int32_t left;  // quads of the current block not yet issued
  int32_t row;   // row of the current block (hi: past the last)
  uint32_t issued;
  int32_t lo, hi;        // the CTA's rows
  const uint32_t* bits;  // which of them need a selection (sched::balanced_range)
  const float4* wbeg;    // checked build: the row's window rounded out to 16 bytes
  const float4* wend;
};

// Whole warp: moves the cursor to the block of its next row with seq_len > k
// (found in the CTA's bitmask).  `ahead` is the descriptor of row `ahead_row`,
// loaded ahead by the caller: used when it is the row needed, which spares a
// wait for global memory.  False past the last.
__device__ __forceinline__ bool cursor_next_row(WCursor& cur, const Params& p, int w, int64_t ahead_row,
                                                const RowRaw& ahead) {
  const int64_t row = sched::next_selected_row(p, cur.bits, cur.lo, cur.hi, (int64_t)cur.row + 1);
  if (row >= cur.hi) {
    cur.row = cur.hi;
    return false;
  }
  int32_t L, st;
  if (row == ahead_row) {
    L = ahead.L;
    st = ahead.start;
  } else if (row_index_ok(p, row)) {
    L = __ldg(p.seq_lens + row);
    st = __ldg(p.row_starts + row);
  } else {
    L = 0;
    st = 0;
  }
  check_row_window(p, L, st);
  cur.row = (int32_t)row;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p.scores + row * p.row_stride + st);
  const int32_t head = (int32_t)((a & 15u) >> 2);
  int64_t q0, q1;
  const int64_t nq = ((int64_t)L + head + 3) >> 2;
  warp_block(nq, w, q0, q1);
  cur.src = reinterpret_cast<const float4*>(a & ~(uintptr_t)15u) + q0;
  cur.left = (int32_t)(q1 - q0);
  if constexpr (kChecked) {
    cur.wbeg = reinterpret_cast<const float4*>(a & ~(uintptr_t)15u);
    cur.wend = cur.wbeg + nq;
  }
  return true;
}

// Whole warp: lane 0 issues the warp's next chunk into stage issued % NS
// (whose previous chunk the warp has taken and fenced).  False past the last row.
template <int NS>
__device__ __forceinline__ bool warp_issue(Ring<NS>& R, WCursor& cur, const Params& p, int w, uint64_t policy,
                                           int64_t ahead_row, const RowRaw& ahead) {
  while (cur.left == 0)
    if (!cursor_next_row(cur, p, w, ahead_row, ahead)) return false;
  const uint32_t s = cur.issued % NS;
  const uint32_t nquads = (uint32_t)min(kWChunkQuads, cur.left);
  if ((threadIdx.x & 31) == 0) {
    if (!in_bounds(cur.src >= cur.wbeg && cur.src + nquads <= cur.wend, kSiteWindowCopy)) {
      mbar_arrive(&R.full[w][s]);  // checked build: the phase completes without the copy
    } else {
      mbar_arrive_expect_tx(&R.full[w][s], nquads * 16u);
      bulk_copy_g2s(&R.st[w][s][0], cur.src, nquads * 16u, &R.full[w][s], policy);
    }
  }
  cur.src += nquads;
  cur.left -= nquads;
  ++cur.issued;
  return true;
}

// ---------------------------------------------------------------------------
// Deferred page transform.  A fast row's emission writes the selected window
// indices j in order; the page transform of section 1 (a load from the page
// table, which comes from L2 -- shared memory leaves little L1) is then done in
// place by each warp for its eighth of the row while the next row streams,
// one position per lane per chunk, its loads issued one chunk ahead, so their
// latency hides behind the stream.  What is left is finished before the next
// fast row's emission and at the end of the kernel.
// ---------------------------------------------------------------------------
struct Deferred {
  int32_t* o;               // output row being transformed (null: none)
  const int32_t* page_row;
  uint32_t next;            // this lane's next position to load; next - 32 and
  uint32_t first, end;      // next - 64 are in the pipeline if in [first, end)
  int32_t ja, jb, pgb;
  int32_t L;                // the row's window length
};

// The indices of the row were written by every warp: a consumer barrier must
// separate that emission from the first deferred_step / deferred_flush.
__device__ __forceinline__ void deferred_start(Deferred& d, int32_t* o, const int32_t* page_row, uint32_t k,
                                               int32_t L) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  d.o = o;
  d.page_row = page_row;
  d.L = L;
  d.first = (uint32_t)((uint64_t)k * w / kWarps) + lane;
  d.next = d.first;
  d.end = (uint32_t)((uint64_t)k * (w + 1) / kWarps);
}

// One step of the pipeline: store the oldest, load the page of the middle,
// load the index of the newest.
__device__ __forceinline__ void deferred_step(Deferred& d, int32_t page_bits) {
  if (d.o == nullptr) return;
  const uint32_t tb = d.next - 64u, ta = d.next - 32u;  // wrap around below 0: out of range
  if (tb >= d.first && tb < d.end) __stcg(d.o + tb, d.pgb * (1 << page_bits) + (d.jb & ((1 << page_bits) - 1)));
  if (ta >= d.first && ta < d.end) {
    d.jb = d.ja;
    d.pgb = in_bounds((uint32_t)d.ja < (uint32_t)d.L, kSitePageRead) ? __ldg(d.page_row + (d.ja >> page_bits)) : 0;
  }
  if (d.next < d.end) d.ja = __ldcg(d.o + d.next);  // written by other warps before a barrier (read from L2)
  d.next += 32u;
}

__device__ __forceinline__ void deferred_flush(Deferred& d, int32_t page_bits) {
  if (d.o == nullptr) return;
  while (d.next < d.end + 64u) deferred_step(d, page_bits);
  d.o = nullptr;
}

// ---------------------------------------------------------------------------
// Fast pass: the warp's block of the row through its ring, fixed threshold.
// ---------------------------------------------------------------------------

// Warp w (of the NW streaming warps) takes its block of the row from its
// ring (NS stages) into its region of S (kCap / NW entries).  With NW ==
// kWarps the regions are the selection's; with more streaming warps their
// counts go to S.scnt and the finishing side merges regions.
//
// The stream loop is kept short: each lane compares its 32 consecutive floats
// with the threshold, the lanes' output positions come from one reduction and
// six ballots (the bits of the lanes' counts), and an admitted element is
// stored as its raw float bits with its window index.  Keys and the fine
// histogram are made afterwards, once per admitted element
// (keys_and_histogram).
//
// A chunk is taken only once its copy has landed.  If a wait gives up
// (`limit_ns`), the warp records it in timed_out and stops taking chunks, for
// this row and every later one: its chunks stay outstanding and their stages
// are not refilled, so no stage ever holds two copies in flight; the kernel's
// exit waits for what is left.  Such a warp marks each of its rows as
// overflowed, so they are finished exactly from global memory.
template <int NS, int NW, int CQ, class E = ElemF32, class AfterChunk>
__device__ __forceinline__ void stream_row_wb(Shared& S, Ring<NS, NW, CQ>& R, int w, const Row& r, int64_t nq,
                                              uint32_t& g, bool& timed_out, uint64_t limit_ns,
                                              AfterChunk&& after_chunk) {
  static_assert(NW == kWarps || NW <= kMaxStreamWarps, "streaming warps");
  constexpr int QPL = CQ / 32;  // quads per lane: 8 (4 KB chunks) or 16 (8 KB chunks)
  constexpr int EPQ = E::kPerQuad;
  constexpr int kBits = EPQ * QPL;  // elements per lane per chunk
  static_assert((QPL == 8 || QPL == 16) && kBits <= 64, "chunk size");
  using Mask = typename std::conditional<kBits <= 32, uint32_t, uint64_t>::type;
  constexpr int kReg = kCap / NW;  // this warp's region
  const int lane = threadIdx.x & 31;
  int64_t q0, q1;
  warp_block_of<NW>(nq, w, q0, q1);
  const float tf = S.rule.tf;
  uint32_t t2 = 0u;  // 16-bit elements: the threshold in both halves of a word
  if constexpr (EPQ == 8) t2 = E::threshold_pair(tf);
  const int rot = lane & 7;  // rotated quad order: the 8 lanes of a load phase hit 8 distinct bank groups
  const uint32_t lt = lanemask_lt();
  uint32_t* rraw = S.bkey + w * kReg;  // raw float bits here; keys after keys_and_histogram
  int32_t* rj = S.bj + w * kReg;
  uint32_t wcnt = 0;
  bool full = false;
  uint32_t s = g % NS, ph = (g / NS) & 1u;
  for (int64_t cq = q0; cq < q1; cq += CQ, ++g) {
    if (timed_out || (!mbar_try_wait(&R.full[w][s], ph) && !mbar_wait_bounded(&R.full[w][s], ph, limit_ns))) {
      timed_out = true;
      if (lane == 0) S.overflow = 1u;  // the row is finished from global memory
      break;
    }
    const float4* st = R.st[w][s];
    // the lane's kBits consecutive elements; bit EPQ*u+c of mr is element
    // EPQ*((u+rot)%QPL)+c
    Mask mr = 0u;
#pragma unroll
    for (int u = 0; u < QPL; ++u) {
      const float4 v = st[QPL * lane + ((u + rot) & (QPL - 1))];
      if constexpr (EPQ == 8) {
        // two elements a packed compare; element 2i is the low half of word i
        const uint32_t wv[4] = {__float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z), __float_as_uint(v.w)};
#pragma unroll
        for (int i = 0; i < 4; ++i) mr |= (Mask)E::ge_pair(wv[i], t2) << (EPQ * u + 2 * i);
      } else {
        float x[EPQ];
        E::decode(v, x);
#pragma unroll
        for (int c = 0; c < EPQ; ++c)
          if (x[c] >= tf) mr |= (Mask)1u << (EPQ * u + c);
      }
    }
    // bit e: element e of the lane's kBits (rotate left by EPQ rot)
    Mask m = rot == 0 ? mr : (Mask)((mr << (EPQ * rot)) | (mr >> (kBits - EPQ * rot)));
    // window index of the lane's element 0 (window indices fit in 32 bits;
    // lanes before the window start get negative ones, masked below)
    const int32_t jb = (int32_t)((cq + QPL * lane) * EPQ - r.head);
    if (cq == 0 || cq + CQ >= q1) {  // the row's first or the block's last chunk
      // keep the window [0, L) and the block's quads [.., q1) (the rest of a
      // partial chunk's stage is stale)
      const int64_t lo = max(-(int64_t)jb, (int64_t)0);
      const int64_t hi = min(min((int64_t)r.L - jb, (q1 - cq - QPL * lane) * EPQ), (int64_t)kBits);
      const Mask below_hi = hi >= kBits ? ~(Mask)0 : (((Mask)1 << (hi > 0 ? hi : 0)) - 1u);
      const Mask from_lo = lo >= kBits ? (Mask)0 : ~(((Mask)1 << lo) - 1u);
      m &= lo >= hi ? (Mask)0 : (below_hi & from_lo);
    }
    if (!full) {
      const uint32_t n = (uint32_t)(kBits <= 32 ? __popc((uint32_t)m) : __popcll((unsigned long long)m));
      const uint32_t tot = __reduce_add_sync(0xFFFFFFFFu, n);
      if (tot != 0u) {
        if (wcnt + tot > (uint32_t)kReg) {
          full = true;
          if (lane == 0) S.overflow = 1u;
        } else {
          // exclusive prefix of n over the lanes, from the bits of n (the
          // low three suffice unless a lane admitted 8 or more; n <= kBits
          // needs up to 6 bits for 32 elements a lane, 7 for 64)
          constexpr int kCountBits = kBits <= 32 ? 6 : 7;
          uint32_t pos = wcnt;
#pragma unroll
          for (int b = 0; b < 3; ++b)
            pos += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, (n >> b) & 1u) & lt) << b;
          if (__any_sync(0xFFFFFFFFu, n >= 8u)) {
#pragma unroll
            for (int b = 3; b < kCountBits; ++b)
              pos += (uint32_t)__popc(__ballot_sync(0xFFFFFFFFu, (n >> b) & 1u) & lt) << b;
          }
          const void* sf = reinterpret_cast<const char*>(st) + 16 * QPL * lane;  // the lane's elements
          // ascending e: window order within the lane; two at a time, so the
          // two loads are in flight together
          Mask mm = m;
          while (mm) {
            const int e0 = (int)(kBits <= 32 ? __ffs((uint32_t)mm) : __ffsll((unsigned long long)mm)) - 1;
            mm &= mm - 1u;
            const int e1 = (int)(kBits <= 32 ? __ffs((uint32_t)mm) : __ffsll((unsigned long long)mm)) - 1;
            const uint32_t x0 = E::bits_at(sf, e0);
            const uint32_t x1 = e1 >= 0 ? E::bits_at(sf, e1) : 0u;
            // the lane's positions lie below wcnt + tot (checked build)
            if (in_bounds(pos < wcnt + tot, kSiteCandidate)) {
              rraw[pos] = x0;
              rj[pos] = jb + e0;
            }
            if (e1 >= 0) {
              if (in_bounds(pos + 1 < wcnt + tot, kSiteCandidate)) {
                rraw[pos + 1] = x1;
                rj[pos + 1] = jb + e1;
              }
              mm &= mm - 1u;
            }
            pos += e1 >= 0 ? 2u : 1u;
          }
          wcnt += tot;
        }
      }
    }
    // the warp is done with the stage: order its reads before the next copy, refill
    fence_proxy_async_smem();
    __syncwarp();
    after_chunk();
    if (++s == (uint32_t)NS) {
      s = 0u;
      ph ^= 1u;
    }
  }
  if (lane == 0) {
    if constexpr (NW == kWarps) {
      S.rbase[w] = (uint32_t)(w * kRegion);
      S.rcnt[w] = wcnt;
    } else {
      S.scnt[w] = wcnt;
    }
  }
}

// The warp that streamed region w, after the stream of a fast row (the
// region's count published by its lane 0): turns the region's raw float bits
// into keys in place and counts them in the fine histogram (hist2, zero
// beforehand; bins of 2^fh_sh keys from fh_tk), keys above its range in
// S.wtop[w].  Touches only region w and hist2 (by atomics); a barrier must
// follow before the selection.
__device__ __forceinline__ void keys_and_histogram(Shared& S, int w) {
  const int lane = threadIdx.x & 31;
  __syncwarp();  // the region's count was written by one lane of this warp
  const uint32_t base = S.rbase[w];
  const uint32_t cnt = in_bounds(base + S.rcnt[w] <= (uint32_t)kCap, kSiteRegion) ? S.rcnt[w] : 0u;
  const uint32_t tk = S.fh_tk, sh = S.fh_sh;
  uint32_t top = 0;
  for (uint32_t i0 = 0; i0 < cnt; i0 += 128) {  // 4 entries a lane, loads issued together
    uint32_t raw[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t i = i0 + 32u * u + (uint32_t)lane;
      raw[u] = i < cnt ? S.bkey[base + i] : 0u;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t i = i0 + 32u * u + (uint32_t)lane;
      if (i < cnt) {
        const uint32_t key = key_of(__uint_as_float(raw[u]));
        S.bkey[base + i] = key;
        const uint32_t fb = (key - tk) >> sh;
        if (fb < (uint32_t)kFineTop)
          atomicAdd(&S.hist2[fb], 1u);
        else
          ++top;
      }
    }
  }
  top = __reduce_add_sync(0xFFFFFFFFu, top);
  if (lane == 0) S.wtop[w] = top;
}

// Rank the next row's admission threshold should reach in this row: about
// m20 / 20 k in a row of the next row's length (with m20 = 23, 1.15 k: the
// binomial noise at that rank is a few percent of k, so the next row still
// admits at least k when its scores are distributed like this row's), capped
// by the buffer.  0 when there is no next row.
constexpr uint32_t kHintMargin20 = 23;
__device__ __forceinline__ uint32_t hint_rank_for(uint32_t k, int32_t L, int32_t next_len,
                                                  uint32_t m20 = kHintMargin20) {
  if (next_len <= 0) return 0u;
  return (uint32_t)min((int64_t)m20 * k * L / (20 * (int64_t)next_len) + 1, (int64_t)kCap);
}

// Fine shift for a row whose threshold key sits about `d` keys below its k-th
// largest: bins of 2^shift keys put the k-th largest near bin 384.
__device__ __forceinline__ uint32_t fine_shift(uint32_t d) {
  const uint32_t x = max(d / 384u, 1u);
  return (uint32_t)(31 - __clz(x));
}

// The fine histogram's bin of rank r (1 <= r <= its total), higher bins
// first.  Thread t owns bins [8 t, 8 t + 8), warp x the range [256 x,
// 256 x + 256); each warp has published, before a barrier, its range total
// (ftot, passed in as `tot`) and per lane the count of its range's bins from
// that lane's on (fsuf).  One warp, no barrier.
struct FinePick {
  uint32_t bin, above, count;  // the bin, the entries in higher bins, its own
};

// Every thread: publishes its warp's scan of `hist` (S.fsuf, S.ftot).  A
// consumer barrier must follow before fine_find reads it.
__device__ __forceinline__ void fine_publish(Shared& S, const uint32_t* hist) {
  const uint4* h4 = reinterpret_cast<const uint4*>(hist) + 2 * threadIdx.x;
  const uint4 a = h4[0], b = h4[1];
  const uint32_t incl = warp_incl_suffix(a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w);
  S.fsuf[threadIdx.x] = incl;
  if ((threadIdx.x & 31) == 0) S.ftot[threadIdx.x >> 5] = incl;
}

__device__ __forceinline__ void fine_totals(const Shared& S, uint32_t (&tot)[kWarps]) {
#pragma unroll
  for (int i = 0; i < kWarps; ++i) tot[i] = S.ftot[i];
}

__device__ __forceinline__ FinePick fine_find(const Shared& S, const uint32_t* hist, const uint32_t (&tot)[kWarps],
                                              uint32_t r) {
  const int lane = threadIdx.x & 31;
  uint32_t run = 0, x = 0, ax = 0;
#pragma unroll
  for (int i = kWarps - 1; i >= 0; --i) {
    const uint32_t prev = run;
    run += tot[i];
    if (prev < r && run >= r) {
      x = (uint32_t)i;
      ax = prev;
    }
  }
  const uint32_t t = x * 32u + (uint32_t)lane;
  const uint4* h4 = reinterpret_cast<const uint4*>(hist) + 2 * t;
  const uint4 a = h4[0], b = h4[1];
  const uint32_t h[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const uint32_t own = a.x + a.y + a.z + a.w + b.x + b.y + b.z + b.w;
  const uint32_t hi = ax + S.fsuf[t] - own;  // entries in bins above this lane's
  const uint32_t yb = __ballot_sync(0xFFFFFFFFu, hi < r && hi + own >= r);
  const int y = yb ? __ffs(yb) - 1 : 0;
  uint32_t bin = 0u, above = 0u, count = 0u;
  uint32_t rr = hi;
#pragma unroll
  for (int i = 7; i >= 0; --i) {
    const uint32_t prev = rr;
    rr += h[i];
    if (prev < r && rr >= r) {
      bin = t * 8u + (uint32_t)i;
      above = prev;
      count = h[i];
    }
  }
  FinePick out;
  out.bin = __shfl_sync(0xFFFFFFFFu, bin, y);
  out.above = __shfl_sync(0xFFFFFFFFu, above, y);
  out.count = __shfl_sync(0xFFFFFFFFu, count, y);
  return out;
}

// Thread 0: the admission rule of the CTA's next row (S.hint).  The row's
// selection proposed `hint` (reaching rank hr, about 1.15 k scaled to the next
// row's length) when hint_ok; otherwise a fast row whose admitted count scales
// to at least 1.05 k of the next row keeps its own rule.  hr == 0: no next row.
__device__ __forceinline__ void publish_hint(Shared& S, uint32_t hr, uint32_t hint_ok, const Rule& hint,
                                             uint32_t hint_sh, bool fast, uint32_t n, uint32_t k, int32_t L) {
  S.hint_valid = 0u;
  if (hr == 0u) return;
  if (hint_ok) {
    S.hint = hint;
    S.hint_sh = hint_sh;
    S.hint_valid = 1u;
  } else if (fast && (uint64_t)n * (uint64_t)S.next_len * 20u >= (uint64_t)21u * k * (uint64_t)L) {
    S.hint = rule_prefix(S.rule.mk, S.rule.tk);
    S.hint_sh = S.fh_sh;
    S.hint_valid = 1u;
  }
}

// Where an emission puts the t-th selected window index j of a row.
// OutRaw: j itself, into the output row in global memory (the page transform
// follows separately; positions below k are the caller's guarantee).
struct OutRaw {
  int32_t* o;
  __device__ __forceinline__ void put(uint32_t q, int32_t j) const { __stcg(o + q, j); }
};

// OutShared: j itself, into a staging row in shared memory.
struct OutShared {
  int32_t* o;  // kBins2 entries
  __device__ __forceinline__ void put(uint32_t q, int32_t j) const {
    if (in_bounds(q < (uint32_t)kBins2, kSiteStaging)) o[q] = j;
  }
};

// Fast rows, entered through a barrier after the stream: the exact k-th
// largest pair from the fine histogram, and the row's selected window indices
// written to out[row] in ascending order.
//
// The bin holding rank k is picked (one barrier); each warp then compacts its
// region in place to the candidates at or above that bin (window order kept),
// counting those above it and gathering those in it; the bin's m <= 32
// candidates are ranked by (key, ~j) in every warp, which settles the k-th
// largest pair T; each warp's output position is the prefix of the warps'
// selected counts, and its compacted candidates are written with ballots.
//
// A split bin of more than 32 candidates that share one key (ties, common
// with bf16 scores) is settled by window order (the lowest indices win); one
// with several keys is narrowed by a second fine level over its entries.
//
// Returns false (uniformly) when the histograms cannot settle it: the rank
// lies above the fine range (before the buffer is touched), or the second
// level's target still holds more than 32 candidates of several keys (the
// regions are then compacted: every entry at or above the first bin kept).
// Also proposes the next row's hint (rank hr) and fine shift.
//
// `out`: where the row's k selected window indices go (OutRaw, OutShared).
template <class Out>
__device__ __forceinline__ bool select_emit_fine(Shared& S, const Out& out, int32_t L, uint32_t n, uint32_t k,
                                                 uint32_t hr) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  uint32_t top = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) top += S.wtop[i];
  if (top >= k) return false;
  const uint32_t tk = S.fh_tk, sh = S.fh_sh;
  const uint32_t r = k - top;                                  // <= n - top, the histogram's total
  const uint32_t r2 = (hr > top && hr <= n) ? hr - top : 0u;
  fine_publish(S, S.hist2);
  cbar();
  uint32_t tot[kWarps];
  fine_totals(S, tot);
  const FinePick pk = fine_find(S, S.hist2, tot, r);
  const FinePick p2 = fine_find(S, S.hist2, tot, r2 != 0u ? r2 : r);  // independent of the first
  const uint32_t lo_key = tk + (pk.bin << sh);
  Rule hint;
  uint32_t hint_ok = 0u, hint_sh = sh;
  if (hr != 0u && hr <= top) {
    hint = rule_prefix(0xFFFFFFFFu, tk + ((uint32_t)kFineTop << sh));
    hint_ok = 1u;
  } else if (r2 != 0u) {
    const uint32_t hk = tk + (p2.bin << sh);
    hint = rule_prefix(0xFFFFFFFFu, hk);
    hint_ok = 1u;
    // ranks k and hr a few bins apart: size the next row's bins from their
    // distance; in the same bin the bins were too wide: halve them
    hint_sh = lo_key > hk ? fine_shift(lo_key - hk) : (sh > 0u ? sh - 1u : 0u);
  }
  const uint32_t rem = r - pk.above;     // rank of the k-th largest inside its bin, 1 <= rem <= count
  const bool split = pk.count != rem;    // only part of the bin is taken
  // more than 32 entries in a split bin: too many to rank in a warp (settled
  // by window order when they share one key, else by a second fine level)
  const bool crowded = split && pk.count > 32u;

  // compaction of the warp's region to the entries at or above the bin, in
  // batches of 4 entries a lane: all read, then written
  uint32_t* rkey = S.bkey + w * kRegion;
  int32_t* rj = S.bj + w * kRegion;
  const uint32_t cnt = S.rcnt[w], bin = pk.bin, lt = lanemask_lt();
  uint32_t wc = 0, cin = 0, kmin = 0xFFFFFFFFu, kmax = 0u;
  for (uint32_t i0 = 0; i0 < cnt; i0 += 4 * 32) {
    uint32_t key[4], bk[4];
    int32_t jj[4];
    uint32_t inb = 0u;  // bit u: entry u lies in the bin
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t i = min(i0 + 32u * u + (uint32_t)lane, (uint32_t)kRegion - 1u);
      key[u] = rkey[i];
      jj[u] = rj[i];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const bool valid = i0 + 32u * u + (uint32_t)lane < cnt;
      const uint32_t fb = (key[u] - tk) >> sh;
      bk[u] = __ballot_sync(0xFFFFFFFFu, valid && fb >= bin);
      inb |= (valid && fb == bin) ? 1u << u : 0u;
    }
    __syncwarp();  // every lane has read its entries before any is overwritten
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if ((bk[u] >> lane) & 1u) {
        const uint32_t q = wc + __popc(bk[u] & lt);
        rkey[q] = key[u];
        rj[q] = jj[u];
      }
      wc += __popc(bk[u]);
    }
    // the bin's entries, when only part of it is taken: gathered for ranking
    // (or, in a crowded bin, counted with their key range)
    const uint32_t nin = split ? (uint32_t)__popc(inb) : 0u;
    if (crowded) {
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if ((inb >> u) & 1u) {
          kmin = min(kmin, key[u]);
          kmax = max(kmax, key[u]);
        }
      cin += __reduce_add_sync(0xFFFFFFFFu, nin);
    } else if (__any_sync(0xFFFFFFFFu, nin != 0u)) {
      uint32_t at = nin ? atomicAdd(&S.res_n, nin) : 0u;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if ((inb >> u) & 1u) {
          if (at < 32u) {  // fewer than count <= 32 are gathered
            S.res_key[at] = key[u];
            S.res_j[at] = jj[u];
            S.res_w[at] = (uint32_t)w;
          }
          ++at;
        }
      cin += __reduce_add_sync(0xFFFFFFFFu, nin);
    }
  }
  if (crowded) {
    kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
    kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  }
  if (lane == 0) {
    S.wtot[w] = wc - cin;  // selected for sure: above the bin, or all of an unsplit bin
    S.rcnt[w] = wc;        // the region is now its compacted entries
    S.wcin[w] = cin;
    S.wkmin[w] = kmin;
    S.wkmax[w] = kmax;
  }
  if (threadIdx.x == 0) publish_hint(S, hr, hint_ok, hint, hint_sh, true, n, k, L);
  cbar();
  // The target: bin t_bin of bins of 2^t_sh keys from tk, of which the t_rem
  // largest pairs are taken.  A crowded bin with several keys is narrowed by a
  // second fine level over its entries: 2^11 sub-bins of it (single keys when
  // the bin is narrower), picked like the first.  Uniform: every warp reads
  // the same published ranges and histograms.
  uint32_t t_sh = sh, t_bin = bin, t_rem = rem, t_count = pk.count, t_cin = cin;
  bool t_split = split, t_crowded = crowded;
  if (crowded) {
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
    for (int x = 0; x < kWarps; ++x) {
      lo = min(lo, S.wkmin[x]);
      hi = max(hi, S.wkmax[x]);
    }
    if (lo != hi) {
      const uint32_t ssh = sh > 11u ? sh - 11u : 0u;
      const uint32_t smask = (1u << (sh - ssh)) - 1u;
      for (int i = threadIdx.x; i < kBins2 / 4; i += kThreads)
        reinterpret_cast<uint4*>(S.hist2)[i] = make_uint4(0u, 0u, 0u, 0u);
      cbar();  // also: every warp has read the published ranges above
      for (uint32_t i = lane; i < wc; i += 32) {
        const uint32_t off = rkey[i] - tk;
        if ((off >> sh) == bin) atomicAdd(&S.hist2[(off >> ssh) & smask], 1u);
      }
      cbar();
      fine_publish(S, S.hist2);
      cbar();
      fine_totals(S, tot);
      const FinePick q2 = fine_find(S, S.hist2, tot, rem);
      t_sh = ssh;
      t_bin = (bin << (sh - ssh)) | q2.bin;
      t_rem = rem - q2.above;  // 1 <= t_rem <= t_count
      t_count = q2.count;
      t_split = t_count != t_rem;
      t_crowded = t_split && t_count > 32u;
      // this warp's entries above the sub-bin and in it (gathered for ranking,
      // or with their key range when crowded)
      uint32_t n_above = 0u, n_in = 0u;
      kmin = 0xFFFFFFFFu;
      kmax = 0u;
      for (uint32_t i0 = 0; i0 < wc; i0 += 32) {
        const uint32_t i = i0 + (uint32_t)lane;
        const uint32_t key = i < wc ? rkey[i] : 0u;
        const uint32_t o2 = (key - tk) >> t_sh;
        const bool ab = i < wc && o2 > t_bin, inb = i < wc && o2 == t_bin;
        n_above += __popc(__ballot_sync(0xFFFFFFFFu, ab));
        n_in += __popc(__ballot_sync(0xFFFFFFFFu, inb));
        if (inb) {
          kmin = min(kmin, key);
          kmax = max(kmax, key);
          if (t_split && !t_crowded) {
            const uint32_t at = atomicAdd(&S.res_n, 1u);
            if (at < 32u) {  // fewer than t_count <= 32 are gathered
              S.res_key[at] = key;
              S.res_j[at] = rj[i];
              S.res_w[at] = (uint32_t)w;
            }
          }
        }
      }
      kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
      kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
      t_cin = t_split ? n_in : 0u;
      if (lane == 0) {
        S.wtot[w] = n_above + (t_split ? 0u : n_in);  // selected for sure
        S.wcin[w] = t_cin;
        S.wkmin[w] = kmin;
        S.wkmax[w] = kmax;
      }
      cbar();
      if (t_crowded) {
        lo = 0xFFFFFFFFu;
        hi = 0u;
#pragma unroll
        for (int x = 0; x < kWarps; ++x) {
          lo = min(lo, S.wkmin[x]);
          hi = max(hi, S.wkmax[x]);
        }
        // still several keys: the generic selection, on the compacted regions
        if (lo != hi) return false;
      }
    }
  }
  uint32_t quota = 0u;  // crowded single-key target: this warp's entries of it that are taken
  if (t_crowded) {
    uint32_t before = 0u;
#pragma unroll
    for (int x = 0; x < kWarps; ++x) before += x < w ? S.wcin[x] : 0u;
    quota = t_rem > before ? min(t_rem - before, t_cin) : 0u;
  }

  // the target's candidates, ranked: the t_rem-th largest pair is the threshold T
  uint64_t T = 0ull;
  uint32_t pos = 0;
  if (t_crowded) {
    // warp x takes min(max(t_rem - (target entries of warps < x), 0), its own)
    uint32_t acc = 0u;
#pragma unroll
    for (int x = 0; x < kWarps; ++x) {
      const uint32_t c = S.wcin[x];
      const uint32_t q = t_rem > acc ? min(t_rem - acc, c) : 0u;
      pos += x < w ? q : 0u;
      acc += c;
    }
  } else if (t_split) {
    const uint32_t m = t_count;  // == S.res_n
    const uint64_t mine = lane < (int)m ? pair_of(S.res_key[lane], S.res_j[lane]) : 0ull;
    const uint32_t mw = lane < (int)m ? S.res_w[lane] : (uint32_t)kWarps;
    uint32_t above = 0;
    for (uint32_t o = 0; o < m; ++o) above += __shfl_sync(0xFFFFFFFFu, mine, o) > mine ? 1u : 0u;
    const uint32_t tb = __ballot_sync(0xFFFFFFFFu, lane < (int)m && above == t_rem - 1u);
    T = __shfl_sync(0xFFFFFFFFu, mine, __ffs(tb) - 1);
    pos = __popc(__ballot_sync(0xFFFFFFFFu, lane < (int)m && mine >= T && mw < (uint32_t)w));
  }
#pragma unroll
  for (int x = 0; x < kWarps; ++x) pos += x < w ? S.wtot[x] : 0u;

  // the compacted entries that are selected, in window order: per batch the
  // ballots first, then the stores
  // o: the output row (or its staging copy)
  bool bad = false;
  uint32_t seen = 0u;  // crowded target: its entries met so far in this warp's region
  for (uint32_t i0 = 0; i0 < wc; i0 += 4 * 32) {
    uint32_t key[4], bm[4];
    int32_t jj[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t i = min(i0 + 32u * u + (uint32_t)lane, (uint32_t)kRegion - 1u);
      key[u] = rkey[i];
      jj[u] = rj[i];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t i = i0 + 32u * u + (uint32_t)lane;
      const uint32_t o2 = (key[u] - tk) >> t_sh;
      const bool above = o2 > t_bin, inb = o2 == t_bin;
      bool take;
      if (t_crowded) {
        // the target's entries in window order: the first `quota` are taken
        const uint32_t bi = __ballot_sync(0xFFFFFFFFu, i < wc && inb);
        take = i < wc && (above || (inb && seen + __popc(bi & lt) < quota));
        seen += __popc(bi);
      } else {
        take = i < wc && (above || (inb && (!t_split || pair_of(key[u], jj[u]) >= T)));
      }
      bm[u] = __ballot_sync(0xFFFFFFFFu, take);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t q = pos + __popc(bm[u] & lt);
      if ((bm[u] >> lane) & 1u) {
        if (q < k) out.put(q, jj[u]);
        bad |= q >= k;
      }
      pos += __popc(bm[u]);
    }
  }
  if (__any_sync(0xFFFFFFFFu, bad) && lane == 0) atomicOr(&g_device_flags, kFlagBadOutputPosition);  // never expected
  return true;
}

// Fast rows whose selection took the generic path: every warp's region is in
// ascending window index and the regions follow each other in warp order, so
// the selected entries' output positions are prefix counts.
// `out`: where the selected window indices go (OutRaw, OutShared).
template <class Out>
__device__ __forceinline__ void emit_ordered(Shared& S, const Out& out, uint32_t k, const Rule sel) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t base = S.rbase[w], cnt = S.rcnt[w];
  const uint32_t lt = lanemask_lt();
  {
    uint32_t c = 0;
    for (uint32_t i = lane; i < cnt; i += 32) c += rule_pass(sel, S.bkey[base + i], S.bj[base + i]) ? 1u : 0u;
    c = __reduce_add_sync(0xFFFFFFFFu, c);
    if (lane == 0) S.wtot[w] = c;
    cbar();
  }
  uint32_t pos = 0;
  for (int i = 0; i < w; ++i) pos += S.wtot[i];
  for (uint32_t i0 = 0; i0 < cnt; i0 += 32) {
    const uint32_t i = i0 + lane;
    bool take = false;
    int32_t j = 0;
    if (i < cnt) {
      j = S.bj[base + i];
      take = rule_pass(sel, S.bkey[base + i], j);
    }
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, take);
    if (take) {
      const uint32_t q = pos + __popc(b & lt);
      if (q < k)
        out.put(q, j);
      else
        atomicOr(&g_device_flags, kFlagBadOutputPosition);  // never expected
    }
    pos += __popc(b);
  }
}

// A row without a hint takes its threshold from a sample of its own
// elements: ns quads spread evenly over the window (ns * kPerQuad elements:
// 4096, or 16384 when 4096 would put fewer than about 128 samples above the
// threshold, i.e. for windows longer than 44.8 k), read from global memory (the same bytes
// stream through the rings right after); lanes outside the window count as
// the lowest key.  The threshold is the sample's rank-R key, R = 1.4 k * n /
// L, so that about 1.4 k of the row's elements reach it; the rank-k key
// (k * n / L) sizes the fine histogram.  Both come from two radix digits of 11
// bits (keys to 2^-13 relative precision), the threshold rounded down to its
// digit.  The second digit reads the sample again (from L2).  It is only a
// guess: if it admits fewer than k elements or overflows a region, the row is
// done again in exact mode.  Entered through a barrier with hist2 zero;
// leaves it zero.
constexpr int kSamples = 4096;
constexpr int kSamplesLong = 16384;
static_assert(kSamples <= kCap, "the 4096-key sample is kept in the candidate buffer");
static_assert(2 * kBins2 <= kCap, "the second digit's histograms use the index buffer");

// Quad s (of ns) of the sample of a window of nq quads.
__device__ __forceinline__ int64_t sample_quad(int64_t s, int64_t ns, int64_t nq) {
  return ((2 * s + 1) * nq) / (2 * ns);
}

template <class E = ElemF32>
__device__ __noinline__ void sample_threshold(Shared& S, const Params& p, const Row r, int64_t nq) {
  constexpr int EPQ = E::kPerQuad;
  const int t = threadIdx.x;
  // samples above the rank-R key: 1.4 k * nsamp / L; at least ~128 of them
  const bool long_sample = (int64_t)r.L * 128 > (int64_t)14 * p.k * kSamples / 10;
  const int nsamp = long_sample ? kSamplesLong : kSamples;
  const int64_t ns = nsamp / EPQ;  // quads sampled
  uint32_t* h1a = reinterpret_cast<uint32_t*>(S.bj);  // second digit under the rank-R digit
  uint32_t* h1b = h1a + kBins2;                        // ... and under the rank-k digit
  for (int b = t; b < 2 * kBins2 / 4; b += kThreads) reinterpret_cast<uint4*>(h1a)[b] = make_uint4(0u, 0u, 0u, 0u);
  // first digit: the top 11 bits of every sampled key (a thread's quads are
  // loaded 8 at a time, all in flight together)
  for (int64_t s0 = t; s0 < ns; s0 += 8 * kThreads) {
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t s = s0 + (int64_t)u * kThreads;
      v[u] = s < ns ? load_window_quad<EPQ>(r, sample_quad(s, ns, nq), kSiteSampleLoad) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int64_t s = s0 + (int64_t)u * kThreads;
      if (s >= ns) continue;
      const int64_t q = sample_quad(s, ns, nq);
      float f[EPQ];
      E::decode(v[u], f);
#pragma unroll
      for (int e = 0; e < EPQ; ++e) {
        const int64_t j = q * EPQ - r.head + e;
        const uint32_t key = (j >= 0 && j < r.L) ? key_of(f[e]) : 0u;
        if (!long_sample) S.bkey[EPQ * s + e] = key;  // kept for the second digit
        atomicAdd(&S.hist2[key >> 21], 1u);
      }
    }
  }
  const int64_t want = (7 * (int64_t)p.k * nsamp) / (5 * (int64_t)r.L) + 1;
  const uint32_t R = (uint32_t)min(want, (int64_t)nsamp);
  const uint32_t Rk = (uint32_t)min((int64_t)p.k * nsamp / r.L + 1, (int64_t)R);
  cbar();
  fine_publish(S, S.hist2);
  cbar();
  uint32_t tot[kWarps];
  fine_totals(S, tot);
  const FinePick a = fine_find(S, S.hist2, tot, R), b = fine_find(S, S.hist2, tot, Rk);
  // second digit: bits 10..20 of the sampled keys in the two chosen bins (the
  // 4096-key sample from shared memory, the larger one read again from L2)
  auto second_digit = [&](uint32_t key) {
    const uint32_t d = key >> 21;
    if (d == a.bin)
      atomicAdd(&h1a[(key >> 10) & (kBins2 - 1)], 1u);
    else if (d == b.bin)
      atomicAdd(&h1b[(key >> 10) & (kBins2 - 1)], 1u);
  };
  if (!long_sample) {
    for (int64_t s = t; s < ns; s += kThreads)  // this thread's own entries
#pragma unroll
      for (int e = 0; e < EPQ; ++e) second_digit(S.bkey[EPQ * s + e]);
  } else {
    for (int64_t s0 = t; s0 < ns; s0 += 8 * kThreads) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t s = s0 + (int64_t)u * kThreads;
        v[u] = s < ns ? load_window_quad<EPQ>(r, sample_quad(s, ns, nq), kSiteSampleLoad)
                      : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int64_t s = s0 + (int64_t)u * kThreads;
        if (s >= ns) continue;
        const int64_t q = sample_quad(s, ns, nq);
        float f[EPQ];
        E::decode(v[u], f);
#pragma unroll
        for (int e = 0; e < EPQ; ++e) {
          const int64_t j = q * EPQ - r.head + e;
          second_digit((j >= 0 && j < r.L) ? key_of(f[e]) : 0u);
        }
      }
    }
  }
  cbar();  // every warp is done with hist2 and the first scan
  for (int i = t; i < kBins2 / 4; i += kThreads) reinterpret_cast<uint4*>(S.hist2)[i] = make_uint4(0u, 0u, 0u, 0u);
  fine_publish(S, h1a);
  cbar();
  fine_totals(S, tot);
  const uint32_t a1 = fine_find(S, h1a, tot, R - a.above).bin;
  uint32_t b1;
  if (b.bin == a.bin) {
    b1 = fine_find(S, h1a, tot, Rk - b.above).bin;
  } else {
    cbar();
    fine_publish(S, h1b);
    cbar();
    fine_totals(S, tot);
    b1 = fine_find(S, h1b, tot, Rk - b.above).bin;
  }
  if (t == 0) {
    const uint32_t thr = (a.bin << 21) | (a1 << 10), tau = (b.bin << 21) | (b1 << 10);
    S.rule = rule_prefix(0xFFFFFC00u, thr);
    S.fh_tk = S.rule.tk;
    S.fh_sh = fine_shift(tau > thr ? tau - thr : 0u);
  }
  cbar();
}

// The pipe kernel's shared memory: its rings, then the row state.
struct PipeSmem {
  Ring<kWStages> ring;
  Shared s;
  sched::RangeSmem range;
  uint64_t never;  // an mbarrier nothing arrives on (kTestUnsatisfiedWait)
};

// Cost floor of a row in the balanced split (elements): the end of a row
// stalls the CTA's stream for about as long as streaming this many elements.
constexpr uint32_t kPipeCostFloor = 24576;

__global__ void __launch_bounds__(kBlock, 2) topk_pipe_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  PipeSmem& M = *reinterpret_cast<PipeSmem*>(smem_raw);
  Shared& S = M.s;
  Ring<kWStages>& R = M.ring;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint32_t k = (uint32_t)p.k;
  const uint64_t policy = l2_evict_first_policy();
  bool timed_out = false;
  if (lane == 0) {
    for (int s = 0; s < kWStages; ++s) mbar_init(&R.full[w][s], 1);
    fence_barrier_init();
  }
  if (tid == 0) {
    S.hint_valid = 0u;
    S.hint_sh = 0u;
    mbar_init(&M.never, 1);
    fence_barrier_init();
  }
  __syncthreads();
  wait_for_producer();
  allow_dependents();
  int64_t lo, hi;
  sched::balanced_range<kThreads>(p, blockIdx.x, gridDim.x, kPipeCostFloor, M.range, lo, hi);
  // each warp starts its ring
  RowRaw nx = {0, 0, 0};
  if (lo < hi) nx = load_row_raw(p, lo);
  WCursor cur;
  cur.src = nullptr;
  cur.left = 0;
  cur.row = (int32_t)lo - 1;
  cur.issued = 0;
  cur.lo = (int32_t)lo;
  cur.hi = (int32_t)hi;
  cur.bits = M.range.bits;
  cur.wbeg = cur.wend = nullptr;
  for (int s = 0; s < kWStages; ++s) warp_issue(R, cur, p, w, policy, lo, nx);
  test_unsatisfied_wait(p, &M.never, timed_out);

  uint32_t g = 0;  // chunks this warp took from its ring
  Deferred dfr;
  dfr.o = nullptr;

  for (int64_t row = lo; row < hi; ++row) {
    const Row r = make_row(p, row, nx);
    const bool has_next = row + 1 < hi;
    if (has_next) nx = load_row_raw(p, row + 1);  // used by the next iteration
    if (r.L <= p.k) {
      emit_whole_window<kThreads>(p, (int32_t)row, r, 0u, 1u);
      continue;
    }
    const int64_t nq = ((int64_t)r.L + r.head + 3) >> 2;
    // ---- row set-up: the threshold (hint, whole row, or sample)
    const bool small = nq * 4 <= kRegion;  // the whole window fits one warp's region
    if (tid == 0) {
      // S.hint_valid is thread 0's own write (after the previous row's
      // selection, with no barrier since): the decision is taken here and
      // published through the barrier below
      const bool hinted = !small && S.hint_valid != 0u;
      S.sample = (!small && !hinted) ? 1u : 0u;
      S.overflow = 0u;
      S.res_n = 0u;
      if (small) {
        S.rule = rule_all();  // every element fits its warp's region
        S.fh_tk = 0u;
        S.fh_sh = 21u;
      } else if (hinted) {
        S.rule = S.hint;
        S.fh_tk = S.hint.tk;
        S.fh_sh = S.hint_sh;
      }
    }
    for (int b = tid; b < kBins2 / 4; b += kThreads) reinterpret_cast<uint4*>(S.hist2)[b] = make_uint4(0u, 0u, 0u, 0u);
    cbar();  // also: every thread is done with the previous row's shared state
    if (S.sample != 0u) sample_threshold(S, p, r, nq);
    stream_row_wb(S, R, w, r, nq, g, timed_out, stream_wait_limit(p), [&] {
      warp_issue(R, cur, p, w, policy, row + 1, nx);
      deferred_step(dfr, p.page_bits);
    });
    deferred_flush(dfr, p.page_bits);  // the previous fast row's transform, if unfinished
    keys_and_histogram(S, w);  // this warp's region, written by this warp
    if (w == 0) {
      // the CTA's next row that needs a selection, for the hint
      int32_t nl = has_next && nx.L > p.k ? nx.L : 0;
      if (nl == 0) {
        const int64_t rr = sched::next_selected_row(p, M.range.bits, lo, hi, row + 2);
        if (rr < hi) nl = __ldg(p.seq_lens + rr);
      }
      if (lane == 0) {
        S.next_len = nl;
        S.hint_rank = hint_rank_for(k, r.L, nl);
      }
    }
    cbar();
    uint32_t n = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) n += S.rcnt[i];
    const bool redo = n < k || S.overflow != 0u;
    const uint32_t hr = S.hint_rank;
    Rule sel, hint;
    uint32_t hint_ok = 0u, hint_sh = S.fh_sh;
    bool emitted = false;
    if (!redo) {
      emitted = select_emit_fine(S, OutRaw{p.out + row * p.k}, r.L, n, k, hr);
      if (!emitted) {
        n = 0u;  // the regions may have been compacted (every entry at or above the k-th key's bin kept)
#pragma unroll
        for (int i = 0; i < kWarps; ++i) n += S.rcnt[i];
        const Selection x = select_buffer(S, n, k, hr);
        sel = x.sel;
        hint = x.hint;
        hint_ok = x.hint_ok;
        hint_sh = (hint_ok && sel.tk > hint.tk) ? fine_shift(sel.tk - hint.tk) : S.fh_sh;
      }
    } else {
      // the threshold was off: stream the row again, from global memory, exactly
      cbar();
      for (int b = tid; b < kBins2 / 4; b += kThreads) reinterpret_cast<uint4*>(S.hist2)[b] = make_uint4(0u, 0u, 0u, 0u);
      if (tid == 0) {
        S.count = 0u;
        S.rule = rule_all();
      }
      cbar();
      stream_row_exact(S, p, r, nq);
      cbar();
      n = S.count;
      set_regions_contiguous(S, n);
      cbar();
      const Selection x = select_buffer(S, n, k, hr);
      sel = x.sel;
      hint = x.hint;
      hint_ok = x.hint_ok;
      hint_sh = (hint_ok && sel.tk > hint.tk) ? fine_shift(sel.tk - hint.tk) : S.fh_sh;
    }
    if (tid == 0 && !emitted) publish_hint(S, hr, hint_ok, hint, hint_sh, !redo, n, k, r.L);
    if (!redo) {
      if (!emitted) emit_ordered(S, OutRaw{p.out + row * p.k}, k, sel);
      if (r.page_row != nullptr) deferred_start(dfr, p.out + row * p.k, r.page_row, k, r.L);  // else j is final
    } else {
      emit_selected(S, p, r, row, sel);
    }
  }

  cbar();  // the last fast row's indices, written by every warp, are visible to all
  deferred_flush(dfr, p.page_bits);

  // Every issued chunk was taken by its warp, so no copy is in flight -- unless
  // a wait gave up; then each warp waits (bounded) for its outstanding copies.
  if (__syncthreads_or(timed_out ? 1 : 0)) {
    if (lane == 0) {
      if (tid == 0) atomicOr(&g_device_flags, kFlagStreamWaitTimeout);
      for (uint32_t c = g; c < cur.issued; ++c) mbar_wait_bounded(&R.full[w][c % kWStages], (c / kWStages) & 1u);
    }
    __syncthreads();
  }
}

}  // namespace pipe
}  // namespace topk
