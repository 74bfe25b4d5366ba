// Row scheduling for the persistent kernels of the packed top-k (sm_103a).
//
// The packed layout (page "[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66%
// 끌어올린 Top-K 커널 최적화 분석", sglang PR #37889, Intro) puts the query rows
// of one request next to each other, in causal order.  Consecutive rows
// therefore have nearly equal window lengths and similar score
// distributions, which is what a threshold carried from one row to the next
// relies on.  So each CTA takes a contiguous range of rows, balanced by an
// estimate of its cost, rather than rows strided over the grid.
//
// A CTA also records which rows of its range need a selection (window longer
// than k) in a shared-memory bitmask, so that skipping the others costs no
// global-memory round trip.
#pragma once

#include "topk_device.cuh"

namespace topk {
namespace sched {

// Rows covered by the balanced split; larger batches are cut into equal counts.
constexpr int32_t kBalanceMaxRows = 1 << 16;
// Bitmask of rows needing a selection: the first kBitRows rows of a range.
constexpr int32_t kBitRows = 8192;
constexpr int32_t kBitWords = kBitRows / 32;

// Estimated cost of a row, in elements streamed.  A row that needs a selection
// costs at least `floor` (the fixed per-row work of selection and emission);
// one that does not costs a fraction of it.
__device__ __forceinline__ uint64_t row_cost(int32_t L, int32_t k, uint32_t floor) {
  if (L > k) return (uint64_t)max((uint32_t)L, floor);
  return (uint64_t)(floor / 8u);
}

__device__ __forceinline__ uint64_t warp_incl_scan64(uint64_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

struct RangeSmem {
  uint64_t warp_sum[32];
  uint32_t lo, hi;
  uint32_t bits[kBitWords];
};

// Rows a thread keeps in registers between the two passes of the split.
constexpr int kRegRows = 32;

// The window lengths of rows [r0, r0 + m) (m <= kRegRows, a multiple of 4; 0
// past n), as independent loads: one round trip.  16-byte loads when the
// rows start on a 16-byte boundary.
__device__ __forceinline__ void load_lengths(const int32_t* seq_lens, int32_t n, int32_t r0, int32_t m,
                                             int32_t (&L)[kRegRows]) {
  const bool vec = ((reinterpret_cast<uintptr_t>(seq_lens + r0) & 15u) == 0u) && r0 + m <= n;
#pragma unroll
  for (int i = 0; i < kRegRows; i += 4) {
    if (i < m) {
      if (vec) {
        const int4 v = __ldg(reinterpret_cast<const int4*>(seq_lens + r0 + i));
        L[i] = v.x; L[i + 1] = v.y; L[i + 2] = v.z; L[i + 3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) L[i + e] = r0 + i + e < n ? __ldg(seq_lens + r0 + i + e) : 0;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) L[i + e] = 0;
    }
  }
}

// Whole CTA (NT threads, entered and left through __syncthreads): the
// contiguous rows [lo, hi) of part `part` of `parts`, and the bitmask of the
// range's rows with a window longer than k.  Every CTA computes the same
// split.  Row i goes to the part that holds the middle of its cost in the
// running sum, so the parts are contiguous and in order, and each row lies in
// exactly one of them.  Thread t takes m consecutive rows; when m <= kRegRows
// their lengths stay in registers between the passes.
template <int NT>
__device__ __forceinline__ void balanced_range(const Params& p, uint32_t part, uint32_t parts, uint32_t floor,
                                               RangeSmem& R, int64_t& lo, int64_t& hi) {
  constexpr int NW = NT / 32;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int32_t n = p.num_rows;
  if (t == 0) {
    R.lo = (uint32_t)n;
    R.hi = (uint32_t)n;
  }
  if (n > kBalanceMaxRows || parts <= 1) {
    if (t == 0) {
      R.lo = (uint32_t)(((int64_t)part * n) / parts);
      R.hi = (uint32_t)(((int64_t)(part + 1) * n) / parts);
    }
  } else {
    const int32_t m = (((n + NT - 1) / NT) + 3) & ~3;  // rows per thread, consecutive
    const int32_t r0 = min(t * m, n), r1 = min(r0 + m, n);
    const bool in_regs = m <= kRegRows;
    int32_t Lr[kRegRows];
    uint64_t s = 0;
    if (in_regs) {
      load_lengths(p.seq_lens, n, r0, m, Lr);
#pragma unroll
      for (int i = 0; i < kRegRows; ++i)
        if (r0 + i < r1) s += row_cost(Lr[i], p.k, floor);
    } else {
      for (int32_t i = r0; i < r1; ++i) s += row_cost(__ldg(p.seq_lens + i), p.k, floor);
    }
    const uint64_t incl = warp_incl_scan64(s);
    if (lane == 31) R.warp_sum[w] = incl;
    __syncthreads();
    uint64_t before = 0, total = 0;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      const uint64_t v = R.warp_sum[i];
      before += i < w ? v : 0ull;
      total += v;
    }
    uint64_t run = before + incl - s;
    if (total == 0) total = 1;
    uint32_t first_lo = (uint32_t)n, first_hi = (uint32_t)n;
    if (in_regs) {
#pragma unroll
      for (int i = 0; i < kRegRows; ++i) {
        if (r0 + i < r1) {
          const uint64_t c = row_cost(Lr[i], p.k, floor);
          const uint64_t owner = min(((run + c / 2) * parts) / total, (uint64_t)(parts - 1));
          if (owner >= part && (uint32_t)(r0 + i) < first_lo) first_lo = (uint32_t)(r0 + i);
          if (owner >= part + 1 && (uint32_t)(r0 + i) < first_hi) first_hi = (uint32_t)(r0 + i);
          run += c;
        }
      }
    } else {
      for (int32_t i = r0; i < r1; ++i) {
        const uint64_t c = row_cost(__ldg(p.seq_lens + i), p.k, floor);
        const uint64_t owner = min(((run + c / 2) * parts) / total, (uint64_t)(parts - 1));
        if (owner >= part && (uint32_t)i < first_lo) first_lo = (uint32_t)i;
        if (owner >= part + 1 && (uint32_t)i < first_hi) first_hi = (uint32_t)i;
        run += c;
      }
    }
    if (first_lo < (uint32_t)n) atomicMin(&R.lo, first_lo);
    if (first_hi < (uint32_t)n) atomicMin(&R.hi, first_hi);
  }
  __syncthreads();
  lo = R.lo;
  hi = max(R.lo, R.hi);
  // bitmask of the range's first kBitRows rows: window longer than k (one
  // word per thread, its 32 loads issued together)
  for (int32_t wd = t; wd < kBitWords; wd += NT) {
    uint32_t b = 0u;
    const int64_t base = lo + (int64_t)wd * 32;
    if (base < hi) {
      int32_t l[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) l[e] = base + e < hi ? __ldg(p.seq_lens + base + e) : 0;
#pragma unroll
      for (int e = 0; e < 32; ++e) b |= (l[e] > p.k ? 1u : 0u) << e;
    }
    R.bits[wd] = b;
  }
  __syncthreads();
}

// Whole warp (uniform result): the first row >= from in [lo, hi) whose window
// is longer than k (SELECTED) or not longer than k (!SELECTED), or hi.  Uses
// the bitmask for the first kBitRows rows of the range and global memory
// beyond them.
template <bool SELECTED>
__device__ __forceinline__ int64_t next_row_where(const Params& p, const uint32_t* bits, int64_t lo, int64_t hi,
                                                  int64_t from) {
  const int lane = threadIdx.x & 31;
  if (from < lo) from = lo;
  const int64_t covered = min(hi, lo + (int64_t)kBitRows);
  // rows below `covered` are found in the bitmask, the others in global memory
  const int64_t global_from = max(from, covered);
  while (from < covered) {
    const int64_t off = from - lo;
    const int64_t wd = (off >> 5) + lane;
    uint32_t b = 0u;
    if (wd < kBitWords) {
      b = SELECTED ? bits[wd] : ~bits[wd];
      // rows at or past the end of the covered part are not in the mask
      const int64_t end = covered - lo - wd * 32;
      if (end < 32) b &= end <= 0 ? 0u : ((1u << end) - 1u);
    }
    if (lane == 0) b &= ~0u << (off & 31);
    const uint32_t nz = __ballot_sync(0xFFFFFFFFu, b != 0u);
    if (nz != 0u) {
      const int src = __ffs(nz) - 1;
      const uint32_t word = __shfl_sync(0xFFFFFFFFu, b, src);
      return lo + (((off >> 5) + src) << 5) + (__ffs(word) - 1);
    }
    from = lo + (((off >> 5) + 32) << 5);
  }
  for (int64_t r0 = global_from; r0 < hi; r0 += 32) {
    const int64_t rr = r0 + lane;
    const int32_t l = rr < hi ? __ldg(p.seq_lens + rr) : 0;
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, rr < hi && ((l > p.k) == SELECTED));
    if (b != 0u) return r0 + (__ffs(b) - 1);
  }
  return hi;
}

__device__ __forceinline__ int64_t next_selected_row(const Params& p, const uint32_t* bits, int64_t lo, int64_t hi,
                                                     int64_t from) {
  return next_row_where<true>(p, bits, lo, hi, from);
}

}  // namespace sched
}  // namespace topk
