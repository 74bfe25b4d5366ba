// Pipelined single-pass kernel of the packed top-k + page transform (sm_103a).
//
// Operation (page "[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66% 끌어올린 Top-K 커널
// 최적화 분석", sglang PR #37889, Intro and sections 1-2): row i's window is
//   scores[i * row_stride + row_starts[i] + j], 0 <= j < seq_lens[i];
// the k largest are kept (a tie goes to the lower j), listed in ascending j and
// mapped through the row's page-table row; -1 pads windows shorter than k.
//
// Design (one CTA per row at a time, two CTAs per SM, rows strided over the
// persistent grid):
//
//  * Load.  The CTA's windows, row after row, stream through a ring of
//    kStages shared-memory stages filled by 1-D TMA bulk copies (16 KB each,
//    L2 evict-first: every byte is read once).  A window is copied from its
//    start rounded down to 16 bytes; lanes before the start and past the end
//    are masked in registers (section 2 of the page, without writing the
//    buffer).  Each stage has a "full" barrier (the copy landed) and an
//    "empty" barrier (all 8 consumer warps took the chunk into registers).
//    A ninth warp only produces: it refills each stage as soon as it is
//    empty, running ahead across rows, so the next row's first chunks are in
//    flight while a row is finished.  The consumer warps synchronise among
//    themselves with named barrier 1, never with the producer.
//
//  * Admission.  Each thread takes 16 floats of a chunk and keeps those at or
//    above the admission threshold, a lower bound on the row's k-th largest
//    key: one float compare per element.  Kept elements (order-preserving
//    key, window index) go to a candidate buffer of kCap entries.
//
//  * Threshold.  When the CTA's previous row gives a hint -- the key prefix
//    that about 1.25 k of its candidates reach, scaled to the new row's
//    length -- the row streams with that fixed threshold and no block-wide
//    synchronisation ("fast" mode): each warp appends to its own region of
//    the buffer at positions from warp ballots, with no shared atomics.  If
//    that admits fewer than k elements or overflows a region, the row is
//    streamed again from global memory in "exact" mode.  Without a hint
//    (first row of a CTA, a much shorter row) the row streams in exact mode
//    from the ring: one shared buffer, a 4096-bin histogram of the key's top
//    12 bits kept as elements arrive, and a threshold that starts at -inf and,
//    whenever a chunk would overflow the buffer, rises to the histogram bin of
//    the k-th largest buffered key, or to the exact k-th largest (key, index)
//    pair.  Any threshold at or below the k-th largest key of the elements
//    seen so far is safe, so no selected element is ever dropped.
//
//  * Selection.  A radix select on the buffer orders candidates by the
//    64-bit pair (key, ~j): larger key first, then lower j.  The candidates'
//    keys share a prefix (the bits where the smallest and largest agree); the
//    digits, 11 bits each, start right below it, so the first level already
//    spreads the candidates over up to 2048 bins.  Levels go on into ~j only
//    for equal keys.  Pairs are unique, so the result is exactly k
//    candidates, whatever the ties.
//
//  * Emission.  The selected window indices are set in a bitmap of the window
//    (reusing the histogram's shared memory, 131072 indices per segment); a
//    block scan of the word popcounts puts the indices, in ascending j, into a
//    staging row; then every thread maps k / 256 of them through the page
//    transform of section 1 (independent loads) and the row leaves with
//    coalesced stores.
#pragma once

#include "topk_device.cuh"

namespace topk {
namespace pipe {

constexpr int kThreads = 256;              // consumer threads (warps 0-7)
constexpr int kWarps = kThreads / 32;
constexpr int kBlock = kThreads + 32;      // + the producer warp
constexpr int kChunkBytes = 16384;
constexpr int kChunkQuads = kChunkBytes / 16;  // 1024
constexpr int kQuadsPerThread = kChunkQuads / kThreads;  // 4: quads tid + u * kThreads
constexpr int kHalfElems = kChunkQuads * 2;    // exact mode admits a chunk in two halves of 2048
constexpr int kStages = 3;
constexpr int kKMax = 2048;
constexpr int kCap = 4096;                 // candidate buffer entries
constexpr int kRegion = kCap / kWarps;     // fast mode: one region of the buffer per warp
constexpr int kBins1 = 4096;               // key bits [20, 32)
constexpr int kBins2 = 2048;               // refinement levels (<= 11 bits)
constexpr int kSegBits = kBins1 * 32;      // bitmap indices per emission segment
constexpr uint32_t kMaskBin = 0xFFF00000u;  // key bits of a level-1 bin
constexpr uint32_t kMaskSub = 0xFFFFFC00u;  // key bits of a level-2 sub-bin

static_assert(kQuadsPerThread == 4, "each thread takes four quads of a chunk");
// After an exact compaction the buffer holds k entries; a half chunk must fit.
static_assert(kCap - kKMax >= kHalfElems, "candidate buffer too small for k + half a chunk");
static_assert(kBins2 >= kKMax, "the output staging row reuses the level-2 histogram");

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

__device__ __forceinline__ Rule rule_bin(uint32_t bin) { return rule_prefix(kMaskBin, bin << 20); }

__device__ __forceinline__ bool rule_pass(const Rule& a, uint32_t key, int32_t j) {
  const uint32_t kk = key & a.mk;
  return kk > a.tk || (kk == a.tk && ((~(uint32_t)j) & a.mj) >= a.tj);
}

// Lowest level-1 bin that can hold an admitted key under rule a.
__device__ __forceinline__ uint32_t rule_low_bin(const Rule& a) { return (a.mk & kMaskBin) ? a.tk >> 20 : 0u; }

struct PickOut {
  uint32_t bin, above, count;  // first target: bin holding rank r, count above it, its count
  uint32_t bin2, has2;         // second target (optional)
  uint32_t total;
};

struct Shared {
  float4 ring[kStages][kChunkQuads];
  uint32_t bkey[kCap];
  int32_t bj[kCap];
  uint32_t hist1[kBins1];  // also the emission bitmap
  uint32_t hist2[kBins2];  // also the output staging row
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint32_t scratch[2][kWarps];
  PickOut pick[2];
  uint32_t wtot[kWarps];
  uint32_t rbase[kWarps], rcnt[kWarps];  // the buffer, as one region per warp (see set_regions_*)
  uint32_t qlist[kWarps][4 * 32];        // fast mode: a warp's quads that may hold candidates
  uint32_t wmin[kWarps], wmax[kWarps];
  uint32_t count;
  uint32_t overflow;  // fast mode: a reservation did not fit
  Rule rule;          // admission rule of the current row
  Rule hint;          // admission rule proposed for the next row
  uint32_t hint_valid;
  uint32_t hint_rank;  // rank the next row's hint should reach in this row (0: none)
  int32_t next_len;    // window length of the CTA's next row that needs a selection
  uint32_t pad_;
};

// Thread 0's cursor over the CTA's chunk sequence: the windows of rows
// blockIdx.x, blockIdx.x + gridDim.x, ... (rows with seq_len <= k have none),
// each cut into kChunkBytes pieces.
struct Cursor {
  const char* src;
  int64_t left;
  int64_t row;
  uint32_t issued;
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

// The producer lane: issues chunk number cur.issued of the sequence into its stage,
// after the stage's previous chunk was taken by every consumer warp.  Returns false
// past the last chunk.
__device__ __forceinline__ bool issue_next(Shared& S, Cursor& cur, const Params& p, uint64_t policy,
                                           bool& timed_out) {
  while (cur.left == 0) {
    if (cur.row >= p.num_rows) return false;
    cur.row += gridDim.x;
    if (cur.row >= p.num_rows) return false;
    const Row r = load_row(p, (int32_t)cur.row);
    if (r.L <= p.k) continue;
    cur.src = reinterpret_cast<const char*>(r.base4);
    cur.left = (((int64_t)r.L + r.head + 3) >> 2) * 16;
  }
  const uint32_t c = cur.issued, s = c % kStages;
  if (c >= (uint32_t)kStages) {
    const uint32_t prev = c - kStages;
    if (!timed_out && !mbar_wait_bounded(&S.empty[s], (prev / kStages) & 1u)) timed_out = true;
  }
  const uint32_t nb = (uint32_t)min((int64_t)kChunkBytes, cur.left);
  mbar_arrive_expect_tx(&S.full[s], nb);
  bulk_copy_g2s(&S.ring[s][0], cur.src, nb, &S.full[s], policy);
  cur.src += nb;
  cur.left -= nb;
  ++cur.issued;
  return true;
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
__device__ __noinline__ uint32_t filter_buffer(Shared& S, uint32_t n, const Rule rule, Par& par) {
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
__device__ __noinline__ Rule select_buffer(Shared& S, uint32_t n, uint32_t r, uint32_t r2, Rule* hint,
                                           uint32_t* hint_ok, Par& par, bool ready = false) {
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
  if (hint_ok) {
    *hint_ok = (r2 != 0u && r2 <= n) ? 1u : 0u;
    *hint = rule_prefix((uint32_t)(HM >> 32), (uint32_t)(HT >> 32));  // the key part: never higher
  }
  return rule_of_pair_prefix(M, T);
}

// The buffer would overflow: raise the threshold.  attempt 0 moves it to the
// level-1 bin of the k-th largest buffered key; attempt 1 (or when that does
// not rise) to the exact k-th largest pair.  n > k entries are buffered.
__device__ __noinline__ void compact(Shared& S, uint32_t n, uint32_t k, int attempt, Par& par) {
  const Rule cur = S.rule;  // read before filter_buffer's first barrier; written after it
  const uint32_t lo = rule_low_bin(cur);
  if (attempt == 0 && !cur.exact) {
    cbar();
    const PickOut p1 = pick_bins<kBins1>(S.hist1, lo, k, 0u, S, par);
    if (p1.bin > lo || cur.mk == 0u) {
      const Rule a = rule_bin(p1.bin);
      filter_buffer(S, n, a, par);
      if (threadIdx.x == 0) S.rule = a;
      cbar();
      return;
    }
  }
  set_regions_contiguous(S, n);
  cbar();
  const Rule a = select_buffer(S, n, k, 0u, nullptr, nullptr, par);
  const uint32_t kept = filter_buffer(S, n, a, par);
  // hist1 must count the buffer exactly again (the bin of the threshold lost entries)
  for (int b = threadIdx.x; b < kBins1; b += kThreads) S.hist1[b] = 0u;
  if (threadIdx.x == 0) S.rule = a;
  cbar();
  for (uint32_t i = threadIdx.x; i < kept; i += kThreads) atomicAdd(&S.hist1[S.bkey[i] >> 20], 1u);
  cbar();
}

// Takes this thread's 16 floats of the row's chunk (quads cq + tid + u * kThreads,
// u < 4; x[4u + v] is element v of quad u): from ring chunk g, or straight
// from global memory.  A ring stage must then be given back with
// release_chunk once the values have been used.
template <bool kRing>
__device__ __forceinline__ void take_chunk(Shared& S, const Row& r, int64_t nq, int64_t cq, uint32_t g,
                                           bool& timed_out, float x[16]) {
  float4 v[kQuadsPerThread];
  if constexpr (kRing) {
    const uint32_t s = g % kStages;
    if (!timed_out && !mbar_wait_bounded(&S.full[s], (g / kStages) & 1u)) timed_out = true;
#pragma unroll
    for (int u = 0; u < kQuadsPerThread; ++u) v[u] = S.ring[s][threadIdx.x + u * kThreads];
  } else {
#pragma unroll
    for (int u = 0; u < kQuadsPerThread; ++u) {
      const int64_t q = cq + threadIdx.x + u * kThreads;
      v[u] = q < nq ? __ldg(r.base4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
#pragma unroll
  for (int u = 0; u < kQuadsPerThread; ++u) {
    x[4 * u] = v[u].x;
    x[4 * u + 1] = v[u].y;
    x[4 * u + 2] = v[u].z;
    x[4 * u + 3] = v[u].w;
  }
}

// Exact mode's view of a chunk: the thread's quads 2h and 2h + 1 (8 floats)
// of half h, read from the ring stage of chunk g (already waited for) or from
// global memory.
template <bool kRing>
__device__ __forceinline__ void take_half(const Shared& S, const Row& r, int64_t nq, int64_t cq, uint32_t g,
                                          int h, float x[8]) {
  float4 v[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int qi = threadIdx.x + (2 * h + u) * kThreads;
    if constexpr (kRing) {
      v[u] = S.ring[g % kStages][qi];
    } else {
      const int64_t q = cq + qi;
      v[u] = q < nq ? __ldg(r.base4 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  x[0] = v[0].x; x[1] = v[0].y; x[2] = v[0].z; x[3] = v[0].w;
  x[4] = v[1].x; x[5] = v[1].y; x[6] = v[1].z; x[7] = v[1].w;
}

// x[e] for a run-time e in [0, 8), as a tree of selects (indexing the array
// with a run-time value would move it to local memory).
__device__ __forceinline__ float pick8(const float x[8], int e) {
  const float a = (e & 1) ? x[1] : x[0], b = (e & 1) ? x[3] : x[2];
  const float c = (e & 1) ? x[5] : x[4], d = (e & 1) ? x[7] : x[6];
  const float lo = (e & 2) ? b : a, hi = (e & 2) ? d : c;
  return (e & 4) ? hi : lo;
}

__device__ __forceinline__ float pick16(const float x[16], int e) {
  const float lo = pick8(x, e & 7), hi = pick8(x + 8, e & 7);
  return (e & 8) ? hi : lo;
}

// Window index of element e of 8 consecutive x whose first element has index
// jb0: elements 0-3 are one quad (index jb0 + e), elements 4-7 the quad
// kThreads further on (index jb0 + 4 * kThreads + e - 4).  index16 extends
// this to the thread's four quads.
__device__ __forceinline__ int32_t index8(int64_t jb0, int e) {
  return (int32_t)(jb0 + (e & 3) + ((e & 4) ? 4 * kThreads : 0));
}

__device__ __forceinline__ int32_t index16(int64_t jb0, int e) {
  return (int32_t)(jb0 + (e & 3) + (int64_t)(e >> 2) * 4 * kThreads);
}

// Gives ring stage g % kStages back to the producer.  The stage's next
// content is written by a TMA copy (the async proxy) while these reads were
// plain shared-memory loads (the generic proxy): each thread orders its reads
// before that write with a proxy fence, after the loaded values have been
// used, and the warp then arrives on the stage's "empty" barrier.
__device__ __forceinline__ void release_chunk(Shared& S, uint32_t g) {
  fence_proxy_async_smem();
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&S.empty[g % kStages]);
}

// Bit e set when element e of 8 consecutive x (laid out as index8) passes
// `rule` and lies in the window [0, L).
__device__ __forceinline__ uint32_t admit_mask(const Rule& rule, const float x[8], int64_t jb0, bool edge,
                                               int32_t L) {
  uint32_t m = 0u;
#pragma unroll
  for (int e = 0; e < 8; ++e) m |= (x[e] >= rule.tf ? 1u : 0u) << e;
  if (edge) {
    uint32_t valid = 0u;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int64_t j = jb0 + (e & 3) + ((e & 4) ? 4 * kThreads : 0);
      valid |= (j >= 0 && j < L ? 1u : 0u) << e;
    }
    m &= valid;
  }
  if (rule.exact && m) {
    for (uint32_t mm = m; mm; mm &= mm - 1u) {
      const int e = __ffs(mm) - 1;
      if (!rule_pass(rule, key_of(pick8(x, e)), index8(jb0, e))) m &= ~(1u << e);
    }
  }
  return m;
}

// Exact mode: appends the flagged elements (8 consecutive x) at pos, pos+1, ...
// and counts them in hist1.
__device__ __forceinline__ void append(Shared& S, const float x[8], uint32_t m, uint32_t pos, int64_t jb0) {
  for (uint32_t mm = m; mm; mm &= mm - 1u) {
    const int e = __ffs(mm) - 1;
    const uint32_t key = key_of(pick8(x, e));
    S.bkey[pos] = key;
    S.bj[pos] = index8(jb0, e);
    ++pos;
    atomicAdd(&S.hist1[key >> 20], 1u);
  }
}

// Fast mode: the row's window through the ring with the fixed rule S.rule
// (a key prefix: x >= rule.tf decides) and no block-wide synchronisation.
// Per chunk each thread compares the maximum of each of its 4 quads with the
// threshold; the warp lists its passing quads (about 1 in 7) in qlist, and
// then each lane takes one listed quad from the stage and appends its
// passing elements to the warp's region of the buffer (kRegion entries) at
// positions from the warp's ballots.  A region that would overflow sets
// S.overflow (the row is then done again in exact mode).
__device__ __forceinline__ void stream_row_fast(Shared& S, const Row& r, int64_t nq, uint32_t& g,
                                                bool& timed_out) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int64_t nch = (nq + kChunkQuads - 1) / kChunkQuads;
  const float tf = S.rule.tf;
  const uint32_t lt = lanemask_lt();
  uint32_t* rkey = S.bkey + w * kRegion;
  int32_t* rj = S.bj + w * kRegion;
  uint32_t* ql = S.qlist[w];
  const float qnan = __uint_as_float(0x7FC00000u);  // fails every comparison
  uint32_t wcnt = 0, kmin = 0xFFFFFFFFu, kmax = 0u;
  bool full = false;
  uint32_t s = g % kStages, ph = (g / kStages) & 1u;
  for (int64_t c = 0; c < nch; ++c) {
    const int64_t cq = c * kChunkQuads;
    if (!mbar_try_wait(&S.full[s], ph) && !timed_out && !mbar_wait_bounded(&S.full[s], ph)) timed_out = true;
    const float4* st = S.ring[s];
    const bool edge = c == 0 || c == nch - 1;
    uint32_t B[kQuadsPerThread];
    bool pass[kQuadsPerThread];
#pragma unroll
    for (int u = 0; u < kQuadsPerThread; ++u) {
      float4 v = st[tid + u * kThreads];
      if (edge) {
        const int64_t j = (cq + tid + u * kThreads) * 4 - r.head;
        if (!(j >= 0 && j < r.L)) v.x = qnan;
        if (!(j + 1 >= 0 && j + 1 < r.L)) v.y = qnan;
        if (!(j + 2 >= 0 && j + 2 < r.L)) v.z = qnan;
        if (!(j + 3 >= 0 && j + 3 < r.L)) v.w = qnan;
      }
      pass[u] = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)) >= tf;  // fmaxf ignores a NaN operand
      B[u] = __ballot_sync(0xFFFFFFFFu, pass[u]);
    }
    const uint32_t P1 = __popc(B[0]), P2 = P1 + __popc(B[1]), P3 = P2 + __popc(B[2]);
    const uint32_t T = P3 + __popc(B[3]);
    if (T != 0u && !full) {
      if (pass[0]) ql[__popc(B[0] & lt)] = (uint32_t)tid;
      if (pass[1]) ql[P1 + __popc(B[1] & lt)] = (uint32_t)tid + kThreads;
      if (pass[2]) ql[P2 + __popc(B[2] & lt)] = (uint32_t)tid + 2 * kThreads;
      if (pass[3]) ql[P3 + __popc(B[3] & lt)] = (uint32_t)tid + 3 * kThreads;
      __syncwarp();
      for (uint32_t base = 0; base < T && !full; base += 32) {
        const uint32_t i = base + lane;
        uint32_t m4 = 0u, qi = 0u;
        float4 q4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < T) {
          qi = ql[i];
          q4 = st[qi];
          const int64_t j = (cq + qi) * 4 - r.head;
          m4 = (q4.x >= tf ? 1u : 0u) | (q4.y >= tf ? 2u : 0u) | (q4.z >= tf ? 4u : 0u) | (q4.w >= tf ? 8u : 0u);
          if (edge) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (!(j + e >= 0 && j + e < r.L)) m4 &= ~(1u << e);
          }
        }
        const int32_t jq = (int32_t)((cq + qi) * 4 - r.head);  // used only for in-window elements
        while (true) {
          const bool has = m4 != 0u;
          const uint32_t b = __ballot_sync(0xFFFFFFFFu, has);
          if (b == 0u) break;
          const uint32_t nb = __popc(b);
          if (wcnt + nb > (uint32_t)kRegion) {
            full = true;
            if (lane == 0) S.overflow = 1u;
            break;
          }
          if (has) {
            const int e = __ffs(m4) - 1;
            m4 &= m4 - 1u;
            const float val = (e & 2) ? ((e & 1) ? q4.w : q4.z) : ((e & 1) ? q4.y : q4.x);
            const uint32_t key = key_of(val);
            const uint32_t pos = wcnt + __popc(b & lt);
            rkey[pos] = key;
            rj[pos] = jq + e;
            kmin = min(kmin, key);
            kmax = max(kmax, key);
          }
          wcnt += nb;
        }
      }
    }
    // every read of the stage is done: give it back
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[s]);
    ++g;
    if (++s == (uint32_t)kStages) {
      s = 0u;
      ph ^= 1u;
    }
  }
  kmin = __reduce_min_sync(0xFFFFFFFFu, kmin);
  kmax = __reduce_max_sync(0xFFFFFFFFu, kmax);
  if (lane == 0) {
    S.rbase[w] = (uint32_t)(w * kRegion);
    S.rcnt[w] = wcnt;
    S.wmin[w] = kmin;
    S.wmax[w] = kmax;
  }
}

// Exact mode: the row's window (from the ring, or from global memory) with a
// rising threshold; the buffer is compacted whenever a half chunk would
// overflow it.  One block-wide vote per half chunk.
template <bool kRing>
__device__ __forceinline__ void stream_row_exact(Shared& S, const Params& p, const Row& r, int64_t nq,
                                                 uint32_t& g, bool& timed_out, Par& par) {
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint32_t k = (uint32_t)p.k;
  const int64_t nch = (nq + kChunkQuads - 1) / kChunkQuads;
  Rule rule = S.rule;
  for (int64_t c = 0; c < nch; ++c) {
    const int64_t cq = c * kChunkQuads;
    if constexpr (kRing) {
      if (!timed_out && !mbar_wait_bounded(&S.full[g % kStages], (g / kStages) & 1u)) timed_out = true;
    }
    const bool edge = c == 0 || c == nch - 1;
#pragma unroll 1
    for (int h = 0; h < 2; ++h) {
      float xh[8];
      take_half<kRing>(S, r, nq, cq, g, h, xh);
      const int64_t jb0 = (cq + tid) * 4 - r.head + (int64_t)h * 8 * kThreads;
      uint32_t m = admit_mask(rule, xh, jb0, edge, r.L);
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
        compact(S, held, k, attempt, par);
        rule = S.rule;
        for (uint32_t mm = m; mm; mm &= mm - 1u) {
          const int e = __ffs(mm) - 1;
          if (!rule_pass(rule, key_of(pick8(xh, e)), index8(jb0, e))) m &= ~(1u << e);
        }
      }
      append(S, xh, m, pos, jb0);
    }
    if constexpr (kRing) {
      release_chunk(S, g);
      ++g;
    }
  }
}

// A row without a hint takes its threshold from kSamples of its own elements:
// kSamples / 4 quads spread evenly over the window, read from global memory
// (the same bytes stream through the ring right after).  The threshold is the
// key prefix of the sample's rank-R element, R = 1.4 k * kSamples / L, so
// that about 1.4 k of the row's elements reach it.  It is only a guess: if it
// admits fewer than k elements or overflows the buffer, the row is done
// again in exact mode.  Windows of at least kSampleMinLen elements only (the
// sampled quads are then distinct).
constexpr int kSamples = 4096;
constexpr int kSampleMinLen = 16384;
static_assert(kSamples <= kCap, "the sample is ranked in the candidate buffer");

__device__ __noinline__ void sample_threshold(Shared& S, const Params& p, const Row& r, int64_t nq, Par& par) {
  constexpr int kSampleQuads = kSamples / 4;
#pragma unroll
  for (int u = 0; u < kSampleQuads / kThreads; ++u) {
    const int s = threadIdx.x + u * kThreads;
    const int64_t q = ((2 * (int64_t)s + 1) * nq) / (2 * kSampleQuads);
    const float4 v = __ldg(r.base4 + q);
    const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t j = q * 4 - r.head + e;
      const bool in = j >= 0 && j < r.L;
      S.bkey[4 * s + e] = in ? key_of(f[e]) : 0u;  // below every real key
      S.bj[4 * s + e] = in ? (int32_t)j : 0;
    }
  }
  set_regions_contiguous(S, kSamples);
  cbar();
  const int64_t want = (7 * (int64_t)p.k * kSamples) / (5 * (int64_t)r.L) + 1;
  const uint32_t rank = (uint32_t)min(want, (int64_t)kSamples);
  const Rule sel = select_buffer(S, kSamples, rank, 0u, nullptr, nullptr, par);
  cbar();
  for (uint32_t b = threadIdx.x; b < (uint32_t)kBins2; b += kThreads) S.hist2[b] = 0u;
  if (threadIdx.x == 0) S.rule = rule_prefix(sel.mk, sel.tk);
  cbar();
}

// Writes the buffer entries that pass `sel` (exactly k of them) in ascending
// window index, through the page transform, to out_row[0, k).
// `clean`: the bitmap (hist1) is already all zero for the first segment.
__device__ __forceinline__ void emit_selected(Shared& S, const Params& p, const Row& r, int64_t row,
                                              const Rule sel, Par& par, bool clean) {
  const int t = threadIdx.x, lane = t & 31;
  const uint32_t rbase = S.rbase[t >> 5], rcnt = S.rcnt[t >> 5];
  uint32_t* bm = S.hist1;
  int32_t* stage = reinterpret_cast<int32_t*>(S.hist2);
  const uint32_t k = (uint32_t)p.k;
  uint32_t out_base = 0;
  for (int64_t seg = 0; seg < r.L; seg += kSegBits) {
    const int32_t seg_lo = (int32_t)seg;
    const int32_t span = (int32_t)min((int64_t)kSegBits, (int64_t)r.L - seg);
    const int32_t nw = (span + 31) >> 5;
    if (seg > 0 || !clean) {
      cbar();  // previous users of the bitmap are done
      for (int i = 4 * t; i < nw; i += 4 * kThreads) *reinterpret_cast<uint4*>(bm + i) = make_uint4(0u, 0u, 0u, 0u);
      cbar();
    }
    for (uint32_t i = lane; i < rcnt; i += 32) {
      const int32_t j = S.bj[rbase + i];
      if (j >= seg_lo && j - seg_lo < span && rule_pass(sel, S.bkey[rbase + i], j))
        atomicOr(&bm[(j - seg_lo) >> 5], 1u << ((j - seg_lo) & 31));
    }
    cbar();
    // warp w owns a run of whole 32-word rounds of the bitmap; in each round
    // lane l takes word round * 32 + l, so the ranks come from warp scans
    const int warp = t >> 5;
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
          stage[pos] = seg_lo + i * 32 + (__ffs(b) - 1);
        else
          atomicOr(&g_device_flags, kFlagBadOutputPosition);  // never expected
        ++pos;
      }
      pos0 += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    cbar();  // S.wtot is read again in the next segment
    out_base += total;
  }
  cbar();
  int32_t* o = p.out + row * p.k;
  constexpr int U = 4;
  for (int i0 = t; i0 < p.k; i0 += kThreads * U) {
    int32_t j[U], pg[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kThreads;
      j[u] = i < p.k ? stage[i] : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) pg[u] = i0 + u * kThreads < p.k ? __ldg(r.page_row + (j[u] >> p.page_bits)) : 0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kThreads;
      if (i < p.k) o[i] = pg[u] * (1 << p.page_bits) + (j[u] & ((1 << p.page_bits) - 1));
    }
  }
}

__global__ void __launch_bounds__(kBlock, 2) topk_pipe_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Shared& S = *reinterpret_cast<Shared*>(smem_raw);
  const int tid = threadIdx.x;
  const uint32_t k = (uint32_t)p.k;
  const uint64_t policy = l2_evict_first_policy();
  bool timed_out = false;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kWarps);
    }
    fence_barrier_init();
    S.hint_valid = 0u;
  }
  __syncthreads();

  if (tid >= kThreads) {
    // ---- producer warp: one lane streams every chunk of the CTA's rows
    Cursor cur;
    cur.src = nullptr;
    cur.left = 0;
    cur.row = (int64_t)blockIdx.x - gridDim.x;
    cur.issued = 0;
    if (tid == kThreads) {
      while (issue_next(S, cur, p, policy, timed_out)) {
      }
    }
    // Every issued chunk is taken by the consumers before they finish, so no
    // copy is in flight at exit -- unless a wait gave up; then wait (bounded)
    // for the last chunks issued.
    if (__syncthreads_or(timed_out ? 1 : 0) && tid == kThreads) {
      atomicOr(&g_device_flags, kFlagStreamWaitTimeout);
      const uint32_t first = cur.issued > (uint32_t)kStages ? cur.issued - kStages : 0u;
      for (uint32_t c = first; c < cur.issued; ++c) mbar_wait_bounded(&S.full[c % kStages], (c / kStages) & 1u);
    }
    return;
  }

  Par par;
  uint32_t g = 0;  // chunks taken from the ring
  // Between rows hist1 (histogram / bitmap) and hist2 (histogram / staging
  // row) are cleared while the next row streams; they start clean.
  for (int b = tid; b < kBins1 / 4; b += kThreads) reinterpret_cast<uint4*>(S.hist1)[b] = make_uint4(0u, 0u, 0u, 0u);
  for (int b = tid; b < kBins2 / 4; b += kThreads) reinterpret_cast<uint4*>(S.hist2)[b] = make_uint4(0u, 0u, 0u, 0u);

  for (int64_t row = blockIdx.x; row < p.num_rows; row += gridDim.x) {
    const Row r = load_row(p, (int32_t)row);
    if (r.L <= p.k) {
      emit_whole_window<kThreads>(p, (int32_t)row, r, 0u, 1u);
      continue;
    }
    const int64_t nq = ((int64_t)r.L + r.head + 3) >> 2;
    // ---- row set-up: threshold from the hint (written at the previous row's end)
    bool fast = S.hint_valid != 0u;
    if (tid == 0) {
      S.count = 0u;
      S.overflow = 0u;
      S.rule = fast ? S.hint : rule_all();
      // the CTA's next row that needs a selection, for the hint
      int32_t nl = 0;
      for (int64_t rr = row + gridDim.x; rr < p.num_rows; rr += gridDim.x) {
        const int32_t l = __ldg(p.seq_lens + rr);
        if (l > p.k) {
          nl = l;
          break;
        }
      }
      S.next_len = nl;
      // rank of about 1.25 k in a row of the next row's length
      S.hint_rank = nl > 0 ? (uint32_t)min((int64_t)5 * k * r.L / (4 * (int64_t)nl) + 1, (int64_t)kCap) : 0u;
    }
    cbar();  // also: every thread is done with the previous row's hist1 / hist2
    for (int b = tid; b < kBins1 / 4; b += kThreads) reinterpret_cast<uint4*>(S.hist1)[b] = make_uint4(0u, 0u, 0u, 0u);
    for (int b = tid; b < kBins2 / 4; b += kThreads) reinterpret_cast<uint4*>(S.hist2)[b] = make_uint4(0u, 0u, 0u, 0u);
    if (!fast && r.L < kSampleMinLen) cbar();  // exact mode counts into hist1 at once
    if (!fast && r.L >= kSampleMinLen) {
      // no hint: estimate a threshold from a sample of the row itself
      sample_threshold(S, p, r, nq, par);
      fast = true;
    }
    if (fast) {
      stream_row_fast(S, r, nq, g, timed_out);
    } else {
      stream_row_exact<true>(S, p, r, nq, g, timed_out, par);
      cbar();
      set_regions_contiguous(S, S.count);
    }
    cbar();
    uint32_t n = 0;
#pragma unroll
    for (int i = 0; i < kWarps; ++i) n += S.rcnt[i];
    const bool redo = n < k || S.overflow;
    // a fast row that stands: hist1 / hist2 untouched since the set-up, key ranges known
    const bool ready = fast && !redo;
    if (redo) {
      // the hint was off: stream the row again, from global memory, exactly
      for (int b = tid; b < kBins1; b += kThreads) S.hist1[b] = 0u;
      cbar();
      if (tid == 0) {
        S.count = 0u;
        S.overflow = 0u;
        S.rule = rule_all();
      }
      cbar();
      stream_row_exact<false>(S, p, r, nq, g, timed_out, par);
      cbar();
      n = S.count;
      set_regions_contiguous(S, n);
      cbar();
    }
    // ---- selection, next row's hint, emission
    Rule hint;
    uint32_t hint_ok = 0u;
    const uint32_t hr = S.hint_rank;
    const Rule sel = select_buffer(S, n, k, hr, &hint, &hint_ok, par, ready);
    if (tid == 0) S.hint_valid = 0u;
    if (tid == 0 && hr != 0u) {
      if (hint_ok) {
        S.hint = hint;
        S.hint_valid = 1u;
      } else if ((uint64_t)n * (uint64_t)S.next_len * 5u >= (uint64_t)6u * k * (uint64_t)r.L) {
        // too few candidates for the rank, but the admitted ones scale to
        // at least 1.2 k in the next row: keep this row's threshold
        S.hint = rule_prefix(S.rule.mk, S.rule.tk);
        S.hint_valid = 1u;
      }
    }
    emit_selected(S, p, r, row, sel, par, ready);
  }

  // (the producer warp joins this last block-wide vote)
  if (__syncthreads_or(timed_out ? 1 : 0) && tid == 0) atomicOr(&g_device_flags, kFlagStreamWaitTimeout);
}

}  // namespace pipe
}  // namespace topk
