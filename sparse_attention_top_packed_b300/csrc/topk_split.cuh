// Warp-specialised kernel of the packed top-k + page transform (sm_103a).
//
// The operation is the one of topk_pipe.cuh (page "[sglang] [AMD ROCm] GLM-5.x
// Prefill 성능을 66% 끌어올린 Top-K 커널 최적화 분석", sglang PR #37889, Intro
// and sections 1-2).  The per-row steps are the same -- blocks of the window
// streamed by 8 warps through TMA rings, admission against a threshold into
// window-ordered regions with a fine histogram, the fine pick, compaction,
// in-bin ranking, ordered emission, page transform -- but they run on two
// groups of warps of one CTA per SM, so that the stream never waits for the
// end of a row:
//
//  * Streaming warps (warps 8 on) only stream: each takes its block of a row
//    through its own ring of TMA stages (two of 8 KB for 32-bit scores, four
//    of 4 KB for 16-bit ones: 128 KB in flight per SM) into its part of one
//    of two row states ("sets"), then hands the set over and goes on with the
//    next row in the other set.  Their loop only compares and appends raw
//    candidates (topk_pipe.cuh, stream_row_wb); for a row shorter than
//    kKeysOnStreamMaxLen they also turn their parts into keys and the fine
//    histogram before the hand-over.  Their rings run ahead on their own: each
//    warp's cursor finds the next row in the CTA's bitmask and has its
//    descriptor loaded a row ahead, so a row change costs no round trip.
//  * Finishing warps (warps 0-7) take a full set, turn its candidates into
//    keys and the fine histogram (for rows of at least kKeysOnStreamMaxLen;
//    joining the streaming warps' parts pairwise into the eight regions of the
//    selection when there are sixteen of them), select and emit its row --
//    the window indices staged in shared memory, then mapped through the page
//    table -- and prepare the set for the row two streamed rows later: its
//    descriptor (read by the streaming warps), its admission rule (the key
//    that about 1.15 k candidates of this row reach, scaled to the new length,
//    or a sample of the new row, or the whole row when small), and a bulk copy
//    of its page-table row into shared memory, so that the page transform
//    reads no global memory.  Descriptors are loaded a row ahead.  While a set
//    is still streaming they emit the rows whose window is not longer than k.
//
// Each CTA takes a contiguous range of rows balanced by cost (topk_sched.cuh).
// With sixteen streaming warps the CTA is launched with 80 registers a thread;
// the streaming warpgroups then give theirs down to 56 and the finishing ones
// take 128 (setmaxnreg).
// Three mbarriers per set carry the hand-overs (streamed / prepared / page row
// staged).  Every wait is bounded; one that gives up raises bit 0 of the
// diagnostics word.
#pragma once

#include "topk_pipe.cuh"
#include "topk_sched.cuh"

namespace topk {
namespace split {

using namespace topk::pipe;

constexpr int kSW = 8;                       // streaming warps (8 or 16)
// Stage size and ring depth per element type: 64 elements a lane per chunk,
// 128 KB in flight per SM.  32-bit: 8 KB stages, 2 of them; 16-bit: 4 KB, 4.
template <class E>
struct Shape {
  static constexpr int kChunk = 16 * 32 * 4 / E::kPerQuad;  // quads per stage
  static constexpr int kStages = (131072 / kSW) / (16 * kChunk);
};
constexpr int kBlockThreads = kThreads + kSW * 32;  // 8 finishing warps, then the streaming warps
constexpr int kPart = kCap / kSW;            // buffer entries of one streaming warp
// Register split (setmaxnreg, per warpgroup of 128 threads): launched with
// kLaunchRegs each; the streaming warpgroups drop to kStreamRegs, the
// finishing ones rise to kFinishRegs.  The sum must not exceed the launch's.
constexpr int kLaunchRegs = 80;
constexpr int kStreamRegs = 56;
constexpr int kFinishRegs = 128;
constexpr bool kRegSplit = kSW > kWarps;
static_assert(!kRegSplit || kSW * 32 * kStreamRegs + kThreads * kFinishRegs <= kBlockThreads * kLaunchRegs,
              "register split exceeds the launch allocation");
static_assert(!kRegSplit || kLaunchRegs * kBlockThreads <= 65536, "launch allocation exceeds the register file");
static_assert(kSW == kWarps || 2 * kPart == kRegion, "two streaming parts make one selection region");
constexpr int kPageStage = 1536;             // page-table entries a set can stage (6 KB)
constexpr uint32_t kHintMargin20Max = 40;    // the hint's widest target: 2 k
constexpr uint32_t kMissSampleRows = 8;      // rows a set samples after a hinted row missed
// Cost floor of a row in the balanced split (elements): the finishing warps
// need about as long per row as the stream takes for this many elements.
constexpr uint32_t kSplitCostFloor = 98304;
// Rows shorter than this (elements) have their candidates turned into keys
// and the fine histogram by the streaming warps, at the end of their stream;
// longer rows leave it to the finishing warps.  Measured on B300: a row's
// finishing takes about 7 us whatever its length, and the stream takes about
// as long for a row of about 68 K elements, so below this length the
// streaming warps would otherwise wait for the finishing warps.  Both sides
// decide from the row's seq_len.  (With sixteen streaming warps the parts are
// merged into regions first, by the finishing warps.)
constexpr int32_t kKeysOnStreamMaxLen = 65536;

__device__ __forceinline__ bool keys_on_stream(int32_t L) { return kSW == kWarps && L < kKeysOnStreamMaxLen; }

// How far the hints of each set are trusted (finishing thread 0's, one
// register: byte b the margin of set b -- the hint's target in twentieths of
// k --, byte 2 + b the rows set b still takes its thresholds from samples).
struct HintAdapt {
  uint32_t v = pipe::kHintMargin20 | (pipe::kHintMargin20 << 8);
  __device__ __forceinline__ uint32_t field(uint32_t i) const { return (v >> (8u * i)) & 0xFFu; }
  __device__ __forceinline__ void set_field(uint32_t i, uint32_t x) {
    v = (v & ~(0xFFu << (8u * i))) | ((x & 0xFFu) << (8u * i));
  }
  __device__ __forceinline__ uint32_t margin(uint32_t b) const { return field(b); }
  __device__ __forceinline__ void set_margin(uint32_t b, uint32_t x) { set_field(b, x); }
  __device__ __forceinline__ uint32_t left(uint32_t b) const { return field(2u + b); }
  __device__ __forceinline__ void set_left(uint32_t b, uint32_t x) { set_field(2u + b, x); }
};

// The row a set is prepared for, as the streaming warps read it.
struct SetRow {
  int64_t row;  // >= the range's end: no more rows
  int32_t L, start, trow, pad_;
};

// What a set's page stage holds.
struct PageStage {
  int32_t trow;    // table row staged (-1: none)
  int32_t off;     // position of page_row[0] in the stage
  int32_t count;   // entries staged from page_row[0] on
  int32_t staged;  // the row the set is prepared for reads its pages from the stage
};

template <class E>
struct SplitSmem {
  using RingT = pipe::Ring<Shape<E>::kStages, kSW, Shape<E>::kChunk>;
  RingT ring;
  pipe::Shared set[2];
  int32_t pages[2][kPageStage];
  SetRow srow[2];
  PageStage pstage[2];
  uint64_t set_full[2];   // streaming -> finishing warps: the set holds its streamed row
  uint64_t set_free[2];   // finishing -> streaming warps: the set is ready for its next row
  uint64_t page_full[2];  // the set's page stage is written (one phase per prepared row)
  uint64_t never;         // an mbarrier nothing arrives on (kTestUnsatisfiedWait)
  sched::RangeSmem range;
};

// Barrier among the streaming warps (the finishing warps use barrier 1).
__device__ __forceinline__ void sbar() { asm volatile("bar.sync 2, %0;" ::"n"(kSW * 32) : "memory"); }

__device__ __forceinline__ bool sbar_or(bool v) {
  uint32_t r;
  asm volatile("{\n\t.reg .pred p, q;\n\t"
               "setp.ne.u32 p, %1, 0;\n\t"
               "bar.red.or.pred q, 2, %2, p;\n\t"
               "selp.u32 %0, 1, 0, q;\n\t}"
               : "=r"(r) : "r"(v ? 1u : 0u), "n"(kSW * 32) : "memory");
  return r != 0u;
}

template <uint32_t N>
__device__ __forceinline__ void regs_raise() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <uint32_t N>
__device__ __forceinline__ void regs_lower() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, bool& timed_out) {
  if (mbar_try_wait(bar, parity)) return true;
  if (timed_out) return false;
  if (!mbar_wait_bounded(bar, parity)) timed_out = true;
  return !timed_out;
}

// 1-D bulk copy global -> shared with the default L2 policy (the page-table
// rows are read by many rows).
__device__ __forceinline__ void bulk_copy_g2s_keep(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// ---------------------------------------------------------------------------
// Streaming warps' cursor over their chunk sequence: the warp's block of each
// row of the CTA's range that needs a selection.  Uniform across the warp.
// ---------------------------------------------------------------------------
struct SCursor {
  const float4* src;
  int32_t left;       // quads of the current block not yet issued
  uint32_t issued;    // chunks issued
  int64_t nrow;       // the row whose block comes next (>= hi: none)
  int32_t nL, nstart; // its descriptor, loaded ahead
  int64_t lo, hi;
  const uint32_t* bits;
  const float4* wbeg;  // checked build: the row's window rounded out to 16 bytes
  const float4* wend;
};

// The descriptor of row c.nrow (in the CTA's range), loaded ahead.
__device__ __forceinline__ void scursor_load_next(SCursor& c, const Params& p) {
  c.nL = 0;
  c.nstart = 0;
  if (c.nrow < c.hi && row_index_ok(p, c.nrow)) {
    c.nL = __ldg(p.seq_lens + c.nrow);
    c.nstart = __ldg(p.row_starts + c.nrow);
  }
}

__device__ __forceinline__ void scursor_init(SCursor& c, const Params& p, int64_t lo, int64_t hi,
                                             const uint32_t* bits) {
  c.src = nullptr;
  c.left = 0;
  c.issued = 0;
  c.lo = lo;
  c.hi = hi;
  c.bits = bits;
  c.wbeg = c.wend = nullptr;
  c.nrow = sched::next_selected_row(p, bits, lo, hi, lo);
  scursor_load_next(c, p);
}

// Moves to the block of row c.nrow and loads the descriptor of the row after
// it (used at the next move).  False past the last row.
template <class E>
__device__ __forceinline__ bool scursor_advance(SCursor& c, const Params& p, int w) {
  if (c.nrow >= c.hi) return false;
  const int64_t row = c.nrow;
  check_row_window(p, c.nL, c.nstart);
  const uintptr_t a = elem_addr<E>(p, row, c.nstart);
  const int32_t head = (int32_t)((a & 15u) / E::kBytes);
  int64_t q0, q1;
  const int64_t nq = ((int64_t)(c.nL > 0 ? c.nL : 0) + head + E::kPerQuad - 1) / E::kPerQuad;
  warp_block_of<kSW>(nq, w, q0, q1);
  c.src = reinterpret_cast<const float4*>(a & ~(uintptr_t)15u) + q0;
  c.left = (int32_t)(q1 - q0);
  if constexpr (kChecked) {
    c.wbeg = reinterpret_cast<const float4*>(a & ~(uintptr_t)15u);
    c.wend = c.wbeg + nq;
  }
  c.nrow = sched::next_selected_row(p, c.bits, c.lo, c.hi, row + 1);
  scursor_load_next(c, p);
  return true;
}

// Whole warp: lane 0 issues the warp's next chunk into stage issued % kStages
// (whose previous chunk the warp has taken and fenced).  False past the last row.
template <class E>
__device__ __forceinline__ bool scursor_issue(typename SplitSmem<E>::RingT& R, SCursor& c, const Params& p, int w,
                                              uint64_t policy) {
  constexpr int kStages = Shape<E>::kStages, kChunk = Shape<E>::kChunk;
  while (c.left == 0)
    if (!scursor_advance<E>(c, p, w)) return false;
  const uint32_t s = c.issued % kStages;
  const uint32_t nquads = (uint32_t)min(kChunk, c.left);
  if ((threadIdx.x & 31) == 0) {
    if (!in_bounds(c.src >= c.wbeg && c.src + nquads <= c.wend, kSiteWindowCopy)) {
      mbar_arrive(&R.full[w][s]);  // checked build: the phase completes without the copy
    } else {
      mbar_arrive_expect_tx(&R.full[w][s], nquads * 16u);
      bulk_copy_g2s(&R.st[w][s][0], c.src, nquads * 16u, &R.full[w][s], policy);
    }
  }
  c.src += nquads;
  c.left -= nquads;
  ++c.issued;
  return true;
}

// ---------------------------------------------------------------------------
// Finishing warps.
// ---------------------------------------------------------------------------

// Finishing threads, entered after a finishing barrier that follows every use
// of set b by its previous row: prepares set b for row R (descriptor d), or
// marks it as the end when R >= hi.  Thread 0 then arrives on set_free[b]
// (done by the caller).  Ends with a finishing barrier.
template <class E>
__device__ __forceinline__ void prepare_set(SplitSmem<E>& M, uint32_t b, const Params& p, int64_t R, const RowRaw& d,
                                            int64_t hi, HintAdapt& ha) {
  pipe::Shared& S = M.set[b];
  if (R >= hi) {
    if (threadIdx.x == 0) M.srow[b].row = hi;
    pipe::cbar();
    return;
  }
  const Row r = make_row<E>(p, R, d);
  const int64_t nq = quads_of<E>(r);
  const bool small = r.L + r.head <= kPart;  // every element fits its streaming warp's part
  if (threadIdx.x == 0) {
    // thread 0's own writes: after a miss the set samples its next rows
    const uint32_t left = ha.left(b);
    const bool hinted = !small && S.hint_valid != 0u && left == 0u;
    S.sample = (!small && !hinted) ? 1u : 0u;
    if (!small && left != 0u) ha.set_left(b, left - 1u);
    S.overflow = 0u;
    S.res_n = 0u;
    if (small) {
      S.rule = pipe::rule_all();
      S.fh_tk = 0u;
      S.fh_sh = 21u;
    } else if (hinted) {
      S.rule = S.hint;
      S.fh_tk = S.hint.tk;
      S.fh_sh = S.hint_sh;
    }
    SetRow sr;
    sr.row = R;
    sr.L = d.L;
    sr.start = d.start;
    sr.trow = d.table_row;
    sr.pad_ = 0;
    M.srow[b] = sr;
    // the page-table row, into the set's page stage (from its 16-byte aligned
    // start; it is reused when the previous row of this set had the same one)
    PageStage& ps = M.pstage[b];
    bool staged = false, copy = false;
    uint32_t bytes = 0;
    uintptr_t a = 0;
    if (r.page_row != nullptr) {
      const int64_t npages = ((int64_t)r.L + (1 << p.page_bits) - 1) >> p.page_bits;
      a = reinterpret_cast<uintptr_t>(r.page_row);
      const int32_t off = (int32_t)((a & 15u) >> 2);
      const int64_t span = (((int64_t)off + npages) * 4 + 15) & ~(int64_t)15;
      if (span <= (int64_t)kPageStage * 4) {
        staged = true;
        if (!(ps.trow == d.table_row && ps.off == off && (int64_t)ps.count >= npages)) {
          copy = true;
          bytes = (uint32_t)span;
          ps.trow = d.table_row;
          ps.off = off;
          ps.count = (int32_t)(span / 4) - off;
        }
      }
    }
    ps.staged = staged ? 1 : 0;
    if (copy) {
      fence_proxy_async_smem();  // earlier reads of the stage come before the copy's writes
      mbar_arrive_expect_tx(&M.page_full[b], bytes);
      bulk_copy_g2s_keep(M.pages[b], reinterpret_cast<const void*>(a & ~(uintptr_t)15u), bytes, &M.page_full[b]);
    } else {
      mbar_arrive(&M.page_full[b]);
    }
  }
  for (int i = threadIdx.x; i < pipe::kBins2 / 4; i += kThreads)
    reinterpret_cast<uint4*>(S.hist2)[i] = make_uint4(0u, 0u, 0u, 0u);
  pipe::cbar();
  if (S.sample != 0u) pipe::sample_threshold<E>(S, p, r, nq);  // ends with a barrier, hist2 zero
}

// Finishing warp w (whole warp): streaming warps 2w and 2w + 1 filled parts
// 2w and 2w + 1 of the buffer (kPart entries each, in window order, part 2w
// first); moves part 2w + 1's entries down to follow part 2w's, which makes
// them region w of the selection, and publishes its count.  The moved range
// only ever goes down, batch by batch, so a batch is read whole before any of
// it is overwritten.
__device__ __forceinline__ void merge_parts(pipe::Shared& S) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t c0 = S.scnt[2 * w], c1 = S.scnt[2 * w + 1];
  uint32_t* key = S.bkey + w * kRegion;
  int32_t* jj = S.bj + w * kRegion;
  if (c0 < (uint32_t)kPart) {
    for (uint32_t i0 = 0; i0 < c1; i0 += 32) {
      const uint32_t i = i0 + (uint32_t)lane;
      uint32_t kv = 0u;
      int32_t jv = 0;
      if (i < c1) {
        kv = key[kPart + i];
        jv = jj[kPart + i];
      }
      __syncwarp();
      if (i < c1) {
        key[c0 + i] = kv;
        jj[c0 + i] = jv;
      }
      __syncwarp();
    }
  }
  if (lane == 0) {
    S.rbase[w] = (uint32_t)(w * kRegion);
    S.rcnt[w] = c0 + c1;
  }
}

// Finishing threads, entered after set b's streamed row R (descriptor d) has
// been handed over: selects and writes row R.  next_len is the window length
// of the row set b serves next (0: none), the target of the hint; `parity`
// the phase of page_full[b] that stages R's pages.  Ends with a finishing
// barrier.
template <class E>
__device__ __forceinline__ void finish_row(SplitSmem<E>& M, uint32_t b, const Params& p, int64_t R, const RowRaw& d,
                                           int32_t next_len, uint32_t parity, bool& timed_out, HintAdapt& ha) {
  pipe::Shared& S = M.set[b];
  const int tid = threadIdx.x;
  const uint32_t k = (uint32_t)p.k;
  const Row r = make_row<E>(p, R, d);
  const int64_t nq = quads_of<E>(r);
  if constexpr (kSW > kWarps) merge_parts(S);
  if (!keys_on_stream(d.L)) pipe::keys_and_histogram(S, tid >> 5);
  if (tid == 0) {
    S.next_len = next_len > p.k ? next_len : 0;
    S.hint_rank = pipe::hint_rank_for(k, r.L, S.next_len, ha.margin(b));
  }
  pipe::cbar();
  int32_t* stage = reinterpret_cast<int32_t*>(S.hist2);  // the row's indices, before the page transform
  const pipe::OutShared out{stage};
  uint32_t n = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) n += S.rcnt[i];
  const bool redo = n < k || S.overflow != 0u;
  const uint32_t hr = S.hint_rank;
  pipe::Rule sel, hint;
  uint32_t hint_ok = 0u, hint_sh = S.fh_sh;
  bool emitted = false;
  if (!redo) {
    emitted = pipe::select_emit_fine(S, out, r.L, n, k, hr);
    if (!emitted) {
      n = 0u;  // the regions may have been compacted
#pragma unroll
      for (int i = 0; i < kWarps; ++i) n += S.rcnt[i];
      const pipe::Selection x = pipe::select_buffer(S, n, k, hr);
      sel = x.sel;
      hint = x.hint;
      hint_ok = x.hint_ok;
      hint_sh = (hint_ok && sel.tk > hint.tk) ? pipe::fine_shift(sel.tk - hint.tk) : S.fh_sh;
    }
  } else {
    // The hint adapts to how far the scores move between this set's rows. A
    // hinted row that admitted fewer than k (its threshold was too high)
    // widens the hint's target by half, up to 2 k, and has the set's next
    // kMissSampleRows rows take their thresholds from samples; a hinted row
    // that overflowed narrows it.  Every hinted row that needs no redo brings
    // it one twentieth of k back toward 1.15 k (below).
    if (tid == 0 && S.sample == 0u) {
      const uint32_t m = ha.margin(b);
      if (S.overflow != 0u) {
        ha.set_margin(b, max(m - m / 4u, pipe::kHintMargin20));
      } else {
        ha.set_margin(b, min(m + m / 2u, kHintMargin20Max));
        ha.set_left(b, kMissSampleRows);
      }
    }
    // the threshold was off: the row again, from global memory, exactly
    pipe::cbar();
    for (int i = tid; i < pipe::kBins2 / 4; i += kThreads)
      reinterpret_cast<uint4*>(S.hist2)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
      S.count = 0u;
      S.rule = pipe::rule_all();
    }
    pipe::cbar();
    pipe::stream_row_exact<E>(S, p, r, nq);
    pipe::cbar();
    n = S.count;
    pipe::set_regions_contiguous(S, n);
    pipe::cbar();
    const pipe::Selection x = pipe::select_buffer(S, n, k, hr);
    sel = x.sel;
    hint = x.hint;
    hint_ok = x.hint_ok;
    hint_sh = (hint_ok && sel.tk > hint.tk) ? pipe::fine_shift(sel.tk - hint.tk) : S.fh_sh;
  }
  if (tid == 0 && !emitted) pipe::publish_hint(S, hr, hint_ok, hint, hint_sh, !redo, n, k, r.L);
  if (tid == 0 && !redo && S.sample == 0u && ha.margin(b) > pipe::kHintMargin20) ha.set_margin(b, ha.margin(b) - 1u);
  if (!redo) {
    if (!emitted) pipe::emit_ordered(S, out, k, sel);
  }
  // the page stage of this row (every prepared row's phase is consumed here,
  // so that the next copy into the stage starts only after this one landed)
  wait_bounded(&M.page_full[b], parity, timed_out);
  pipe::cbar();  // the staged row is complete
  if (!redo) {
    // page transform (section 1 of the page): each thread 8 positions, the
    // index reads, the page reads and the stores each issued together
    constexpr int U = kKMax / kThreads;
    int32_t* o = p.out + R * p.k;
    const int32_t* pr = r.page_row;
    const PageStage ps = M.pstage[b];
    const int32_t* pst = M.pages[b] + ps.off;
    const int32_t pb = p.page_bits, pm = (1 << pb) - 1;
    int32_t jv[U], pg[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = tid + u * kThreads;
      jv[u] = t < (int)k ? stage[t] : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = tid + u * kThreads;
      // a staged index is always inside the window; the test only keeps a
      // broken hand-over from reading outside the page-table row
      bool ok = t < (int)k && pr != nullptr && (uint32_t)jv[u] < (uint32_t)r.L;
      if constexpr (kChecked) {
        if (t < (int)k && pr != nullptr) {
          ok = in_bounds((uint32_t)jv[u] < (uint32_t)r.L, kSitePageRead);
          if (ok && ps.staged)
            ok = in_bounds((jv[u] >> pb) < ps.count && ps.off + (jv[u] >> pb) < kPageStage, kSitePageStage);
        }
      }
      pg[u] = ok ? (ps.staged ? pst[jv[u] >> pb] : __ldg(pr + (jv[u] >> pb))) : 0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = tid + u * kThreads;
      if (t < (int)k) __stcg(o + t, pr != nullptr ? pg[u] * (1 << pb) + (jv[u] & pm) : jv[u]);
    }
  } else {
    pipe::emit_selected(S, p, r, R, sel);  // final values, straight to the output
  }
  pipe::cbar();  // every finishing thread is done with S
}

// Whole warp: this warp's positions of a row whose window is not longer than
// k (every index taken, -1 past the window).
__device__ __forceinline__ void emit_short_row(const Params& p, int64_t row) {
  const Row r = make_row(p, row, load_row_raw(p, row));
  emit_whole_window<kThreads>(p, (int32_t)row, r, 0u, 1u);
}

// Whole warp: waits for the phase `parity` of bar; while it is incomplete the
// warp emits the range's rows that need no selection (`sh`: the next one).
__device__ __forceinline__ void wait_emitting(uint64_t* bar, uint32_t parity, bool& timed_out, const Params& p,
                                              const uint32_t* bits, int64_t lo, int64_t hi, int64_t& sh) {
  while (sh < hi) {
    if (__any_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) break;
    emit_short_row(p, sh);
    sh = sched::next_row_where<false>(p, bits, lo, hi, sh + 1);
  }
  wait_bounded(bar, parity, timed_out);
}

template <class E>
__global__ void __launch_bounds__(kBlockThreads, 1) topk_split_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SplitSmem<E>& M = *reinterpret_cast<SplitSmem<E>*>(smem_raw);
  constexpr int kStages = Shape<E>::kStages;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool finishing = warp < kWarps;
  bool timed_out = false;
  if (!finishing && lane == 0)
    for (int s = 0; s < kStages; ++s) mbar_init(&M.ring.full[warp - kWarps][s], 1);
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&M.set_full[b], 1);
      mbar_init(&M.set_free[b], 1);
      mbar_init(&M.page_full[b], 1);
      M.set[b].hint_valid = 0u;
      M.set[b].hint_sh = 0u;
      M.pstage[b].trow = -1;
      M.pstage[b].off = 0;
      M.pstage[b].count = 0;
      M.pstage[b].staged = 0;
    }
    mbar_init(&M.never, 1);
  }
  if (lane == 0) fence_barrier_init();
  __syncthreads();
  wait_for_producer();
  allow_dependents();
  int64_t lo, hi;
  sched::balanced_range<kBlockThreads>(p, blockIdx.x, gridDim.x, kSplitCostFloor, M.range, lo, hi);
  const uint32_t* bits = M.range.bits;

  uint32_t g = 0;  // streaming warps: chunks taken from the ring
  SCursor cur;
  cur.issued = 0;
  uint32_t page_armed[2] = {0u, 0u}, page_seen[2] = {0u, 0u};  // finishing thread 0: page_full phases

  if (finishing) {
    // ---- finishing warps
    if constexpr (kRegSplit) regs_raise<kFinishRegs>();
    int64_t rc = sched::next_selected_row(p, bits, lo, hi, lo);
    int64_t rn = rc < hi ? sched::next_selected_row(p, bits, lo, hi, rc + 1) : hi;
    RowRaw dc = {0, 0, 0}, dn = {0, 0, 0};
    if (rc < hi) dc = load_row_raw(p, rc);
    if (rn < hi) dn = load_row_raw(p, rn);
    // the first two streamed rows' sets
    HintAdapt ha;  // thread 0's
    prepare_set(M, 0u, p, rc, dc, hi, ha);
    if (tid == 0) {
      if (rc < hi) ++page_armed[0];
      mbar_arrive(&M.set_free[0]);
    }
    if (rc < hi) {
      prepare_set(M, 1u, p, rn, dn, hi, ha);
      if (tid == 0) {
        if (rn < hi) ++page_armed[1];
        mbar_arrive(&M.set_free[1]);
      }
    }
    int64_t sh = sched::next_row_where<false>(p, bits, lo, hi, lo);  // next row needing no selection
    for (uint32_t s = 0; rc < hi; ++s) {
      const uint32_t b = s & 1u, par = (s >> 1) & 1u;
      const int64_t r2 = rn < hi ? sched::next_selected_row(p, bits, lo, hi, rn + 1) : hi;
      RowRaw d2 = {0, 0, 0};
      if (r2 < hi) d2 = load_row_raw(p, r2);  // in flight while the set streams
      wait_emitting(&M.set_full[b], par, timed_out, p, bits, lo, hi, sh);
      finish_row(M, b, p, rc, dc, r2 < hi ? d2.L : 0, par, timed_out, ha);
      if (tid == 0) ++page_seen[b];
      prepare_set(M, b, p, r2, d2, hi, ha);
      if (tid == 0) {
        if (r2 < hi) ++page_armed[b];
        mbar_arrive(&M.set_free[b]);
      }
      rc = rn;
      dc = dn;
      rn = r2;
      dn = d2;
    }
    while (sh < hi) {  // rows needing no selection not yet emitted
      emit_short_row(p, sh);
      sh = sched::next_row_where<false>(p, bits, lo, hi, sh + 1);
    }
  } else {
    // ---- streaming warps
    if constexpr (kRegSplit) regs_lower<kStreamRegs>();
    const int sw = warp - kWarps;
    const uint64_t policy = l2_evict_first_policy();
    scursor_init(cur, p, lo, hi, bits);
    for (int s = 0; s < kStages; ++s) scursor_issue<E>(M.ring, cur, p, sw, policy);
    test_unsatisfied_wait(p, &M.never, timed_out);
    for (uint32_t s = 0;; ++s) {
      const uint32_t b = s & 1u;
      wait_bounded(&M.set_free[b], (s >> 1) & 1u, timed_out);
      const SetRow sr = M.srow[b];
      if (sbar_or(sr.row >= hi || sr.row < lo)) break;  // uniform over the streaming warps
      const Row r = make_row<E>(p, sr.row, RowRaw{sr.L, sr.start, sr.trow});
      const int64_t nq = quads_of<E>(r);
      stream_row_wb<kStages, kSW, Shape<E>::kChunk, E>(M.set[b], M.ring, sw, r, nq, g, timed_out, stream_wait_limit(p),
                                                      [&] { scursor_issue<E>(M.ring, cur, p, sw, policy); });
      if (keys_on_stream(sr.L)) pipe::keys_and_histogram(M.set[b], sw);
      sbar();  // every streaming warp has written its region
      if (tid == kThreads) mbar_arrive(&M.set_full[b]);
    }
  }

  // Every issued chunk was taken, and every staged page row waited for --
  // unless a wait gave up; then each waits (bounded) for what is outstanding.
  if (__syncthreads_or(timed_out ? 1 : 0)) {
    if (tid == 0) {
      atomicOr(&g_device_flags, kFlagStreamWaitTimeout);
      for (int b = 0; b < 2; ++b)
        for (uint32_t c = page_seen[b]; c < page_armed[b]; ++c) mbar_wait_bounded(&M.page_full[b], c & 1u);
    }
    if (!finishing && lane == 0)
      for (uint32_t c = g; c < cur.issued; ++c)
        mbar_wait_bounded(&M.ring.full[warp - kWarps][c % kStages], (c / kStages) & 1u);
    __syncthreads();
  }
}

}  // namespace split
}  // namespace topk
