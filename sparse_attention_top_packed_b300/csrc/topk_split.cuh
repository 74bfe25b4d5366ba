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
//  * Streaming warps (warps 8-15) only stream: each takes its block of a row
//    through its own ring of 4 stages of 4 KB (128 KB in flight per SM) into
//    one of two row states ("sets"), then hands the set over and goes on with
//    the CTA's next row in the other set.
//  * Finishing warps (warps 0-7) take a full set, select and emit its row --
//    the window indices staged in shared memory, then mapped through the page
//    table with independent loads and written out -- and prepare the set for
//    the row two streamed rows later: its admission rule comes from this row
//    (the key that about 1.25 k candidates reach, scaled to the new length), or
//    from a sample of that row taken right here, or the whole row when small.
//    They also emit the rows whose window is not longer than k.
//
// Two mbarriers per set carry the hand-over (streamed / prepared).  Every wait
// is bounded; one that gives up raises bit 0 of the diagnostics word.
#pragma once

#include "topk_pipe.cuh"

namespace topk {
namespace split {

using namespace topk::pipe;

constexpr int kStages = 4;                   // the streaming warps' ring depth
constexpr int kBlockThreads = 2 * kThreads;  // 8 finishing warps, then 8 streaming warps

struct SplitSmem {
  pipe::Ring<kStages> ring;
  pipe::Shared set[2];
  uint64_t set_full[2];  // streaming -> finishing warps: the set holds its streamed row
  uint64_t set_free[2];  // finishing -> streaming warps: the set is ready for its next row
};

// Barrier among the 8 streaming warps (the finishing warps use barrier 1).
__device__ __forceinline__ void sbar() { asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory"); }

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, bool& timed_out) {
  if (mbar_try_wait(bar, parity)) return true;
  if (timed_out) return false;
  if (!mbar_wait_bounded(bar, parity)) timed_out = true;
  return !timed_out;
}

// All finishing threads (uniform): the CTA's first row at or after `from`,
// stepping by the grid, whose window is longer than k; num_rows when none.
__device__ __forceinline__ int64_t next_streamed(const Params& p, int64_t from) {
  const int lane = threadIdx.x & 31;
  for (int64_t r0 = from; r0 < p.num_rows; r0 += 32 * (int64_t)gridDim.x) {
    const int64_t rr = r0 + (int64_t)lane * gridDim.x;
    const int32_t l = rr < p.num_rows ? __ldg(p.seq_lens + rr) : 0;
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, l > p.k);
    if (b != 0u) return r0 + (int64_t)(__ffs(b) - 1) * gridDim.x;
  }
  return p.num_rows;
}

// Finishing threads, entered after a finishing barrier that follows every use
// of S by its previous row: S's admission rule for row R -- the hint S holds,
// the whole row, or a sample of it -- with the histogram cleared.  Ends with a
// finishing barrier.
__device__ __forceinline__ void prepare_set(pipe::Shared& S, const Params& p, int64_t R) {
  const Row r = load_row(p, (int32_t)R);
  const int64_t nq = ((int64_t)r.L + r.head + 3) >> 2;
  const bool small = nq * 4 <= kRegion;  // every element fits its warp's region
  if (threadIdx.x == 0) {
    const bool hinted = !small && S.hint_valid != 0u;  // thread 0's own write
    S.sample = (!small && !hinted) ? 1u : 0u;
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
  }
  for (int b = threadIdx.x; b < pipe::kBins2 / 4; b += kThreads)
    reinterpret_cast<uint4*>(S.hist2)[b] = make_uint4(0u, 0u, 0u, 0u);
  pipe::cbar();
  if (S.sample != 0u) pipe::sample_threshold(S, p, r, nq);  // ends with a barrier, hist2 zero
}

// Finishing threads, entered after S's streamed row R has been handed over:
// selects and writes row R.  R2 is the row S serves next (num_rows: none),
// the target of the hint.  Ends with a finishing barrier.
__device__ __forceinline__ void finish_row(pipe::Shared& S, const Params& p, int64_t R, int64_t R2) {
  const int tid = threadIdx.x;
  const uint32_t k = (uint32_t)p.k;
  const Row r = load_row(p, (int32_t)R);
  const int64_t nq = ((int64_t)r.L + r.head + 3) >> 2;
  if (tid == 0) {
    const int32_t nl = R2 < p.num_rows ? __ldg(p.seq_lens + R2) : 0;
    S.next_len = nl > p.k ? nl : 0;
    // rank of about 1.25 k in a row of the next length
    S.hint_rank = S.next_len > 0
                      ? (uint32_t)min((int64_t)5 * k * r.L / (4 * (int64_t)S.next_len) + 1, (int64_t)kCap)
                      : 0u;
  }
  pipe::cbar();
  uint32_t n = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) n += S.rcnt[i];
  const bool redo = n < k || S.overflow != 0u;
  const uint32_t hr = S.hint_rank;
  int32_t* stage = reinterpret_cast<int32_t*>(S.hist2);  // the row's indices, before the page transform
  pipe::Rule sel, hint;
  uint32_t hint_ok = 0u, hint_sh = S.fh_sh;
  bool emitted = false;
  if (!redo) {
    emitted = pipe::select_emit_fine<true>(S, stage, r.L, n, k, hr);
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
    // the threshold was off: the row again, from global memory, exactly
    pipe::cbar();
    for (int b = tid; b < pipe::kBins2 / 4; b += kThreads)
      reinterpret_cast<uint4*>(S.hist2)[b] = make_uint4(0u, 0u, 0u, 0u);
    if (tid == 0) {
      S.count = 0u;
      S.rule = pipe::rule_all();
    }
    pipe::cbar();
    pipe::stream_row_exact(S, p, r, nq);
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
  if (!redo) {
    if (!emitted) pipe::emit_ordered(S, stage, k, sel);
    pipe::cbar();  // the staged row is complete
    // page transform (section 1 of the page): each thread 8 positions, the
    // index reads, the page loads and the stores each issued together
    constexpr int U = kKMax / kThreads;
    int32_t* o = p.out + R * p.k;
    const int32_t* pr = r.page_row;
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
      pg[u] = (t < (int)k && pr != nullptr && (uint32_t)jv[u] < (uint32_t)r.L) ? __ldg(pr + (jv[u] >> pb)) : 0;
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

__global__ void __launch_bounds__(kBlockThreads, 1) topk_split_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SplitSmem& M = *reinterpret_cast<SplitSmem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool finishing = warp < kWarps;
  bool timed_out = false;
  if (!finishing && lane == 0)
    for (int s = 0; s < kStages; ++s) mbar_init(&M.ring.full[warp - kWarps][s], 1);
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(&M.set_full[b], 1);
      mbar_init(&M.set_free[b], 1);
      M.set[b].hint_valid = 0u;
      M.set[b].hint_sh = 0u;
    }
  }
  if (lane == 0) fence_barrier_init();
  __syncthreads();

  uint32_t g = 0;  // streaming warps: chunks taken from the ring
  WCursor cur;
  cur.src = nullptr;
  cur.left = 0;
  cur.row = (int32_t)blockIdx.x - (int32_t)gridDim.x;
  cur.issued = 0;

  if (finishing) {
    // ---- finishing warps
    int64_t rcur = next_streamed(p, blockIdx.x);
    int64_t rnext = rcur < p.num_rows ? next_streamed(p, rcur + gridDim.x) : p.num_rows;
    // the first two streamed rows' rules
    if (rcur < p.num_rows) {
      prepare_set(M.set[0], p, rcur);
      if (tid == 0) mbar_arrive(&M.set_free[0]);
    }
    if (rnext < p.num_rows) {
      prepare_set(M.set[1], p, rnext);
      if (tid == 0) mbar_arrive(&M.set_free[1]);
    }
    uint32_t s = 0;  // streamed rows finished
    for (int64_t row = blockIdx.x; row < p.num_rows; row += gridDim.x) {
      if (row != rcur) {  // a window not longer than k: every index, no selection
        const Row r = load_row(p, (int32_t)row);
        emit_whole_window<kThreads>(p, (int32_t)row, r, 0u, 1u);
        continue;
      }
      const uint32_t b = s & 1u;
      wait_bounded(&M.set_full[b], (s >> 1) & 1u, timed_out);
      const int64_t r2 = rnext < p.num_rows ? next_streamed(p, rnext + gridDim.x) : p.num_rows;
      finish_row(M.set[b], p, rcur, r2);
      if (r2 < p.num_rows) {
        prepare_set(M.set[b], p, r2);
        if (tid == 0) mbar_arrive(&M.set_free[b]);
      }
      ++s;
      rcur = rnext;
      rnext = r2;
    }
  } else {
    // ---- streaming warps
    const int sw = warp - kWarps;
    const uint64_t policy = l2_evict_first_policy();
    RowRaw nx = load_row_raw(p, blockIdx.x);  // the grid never exceeds num_rows
    for (int s = 0; s < kStages; ++s) warp_issue(M.ring, cur, p, sw, policy, blockIdx.x, nx);
    Deferred none;
    none.o = nullptr;
    uint32_t s = 0;  // streamed rows handed over
    for (int64_t row = blockIdx.x; row < p.num_rows; row += gridDim.x) {
      const Row r = make_row(p, row, nx);
      if (row + gridDim.x < p.num_rows) nx = load_row_raw(p, row + gridDim.x);
      if (r.L <= p.k) continue;
      const uint32_t b = s & 1u;
      wait_bounded(&M.set_free[b], (s >> 1) & 1u, timed_out);
      const int64_t nq = ((int64_t)r.L + r.head + 3) >> 2;
      stream_row_wb(M.set[b], M.ring, sw, p, r, nq, g, cur, policy, timed_out, none, row + gridDim.x, nx);
      sbar();  // every streaming warp has written its region
      if (tid == kThreads) mbar_arrive(&M.set_full[b]);
      ++s;
    }
  }

  // Every issued chunk was taken -- unless a wait gave up; then each
  // streaming warp waits (bounded) for its outstanding copies.
  if (__syncthreads_or(timed_out ? 1 : 0)) {
    if (tid == 0) atomicOr(&g_device_flags, kFlagStreamWaitTimeout);
    if (!finishing && lane == 0)
      for (uint32_t c = g; c < cur.issued; ++c)
        mbar_wait_bounded(&M.ring.full[warp - kWarps][c % kStages], (c / kStages) & 1u);
    __syncthreads();
  }
}

}  // namespace split
}  // namespace topk
