// Kernels of the packed top-k + page transform (sm_103a).
//
//   topk_multipass_kernel  one CTA per row (grid-strided): a 12-bit histogram
//                          of the whole window, then 10-bit refinement levels
//                          on the keys that share the chosen prefix, then the
//                          ordered emission -- every pass straight from global
//                          memory.  Simple and always exact.
//   topk_stream_kernel     persistent CTAs (or clusters of CTAs sharing a row)
//                          that stream every window once from HBM through a
//                          ring of TMA bulk copies into shared memory.  While
//                          streaming, a running lower bound on the k-th largest
//                          key (a histogram bin edge that can only rise) drops
//                          almost every element at a single compare; the few
//                          that pass are appended, in window order, to a list
//                          in shared memory.  The radix select then runs on
//                          that list.  A row whose list cannot hold its
//                          candidates falls back to the multipass procedure.
#pragma once

#include "topk_device.cuh"

namespace topk {

__device__ __forceinline__ bool row_is_whole(const Row& r, int32_t k) { return r.L <= k; }

// ---------------------------------------------------------------------------
// Multipass kernel.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads, 2) topk_multipass_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SelectShared& S = *reinterpret_cast<SelectShared*>(smem_raw);
  ScanParity par;
  for (int64_t row = blockIdx.x; row < p.num_rows; row += gridDim.x) {
    const Row r = load_row(p, (int32_t)row);
    if (row_is_whole(r, p.k)) {
      emit_whole_window(p, (int32_t)row, r, 0u, 1u);
      continue;
    }
    const Part part = part_of(r, 0u, 1u);
    select_from_global<1>(p, (int32_t)row, r, part, S, par);
  }
}

// ---------------------------------------------------------------------------
// Streaming kernel.
// ---------------------------------------------------------------------------
constexpr int kChunkFloats = kThreads * 8;  // one chunk = one tile: 8 floats per thread
constexpr int kChunkBytes = kChunkFloats * 4;
constexpr int kStages = 3;
constexpr int kCap = 4096;  // candidate list entries (>= k plus the threshold bucket)

// Thread 0's position in the chunk sequence (kept in shared memory so that the
// other 511 threads do not hold it in registers).
struct ProducerState {
  int64_t row;
  int64_t bytes;
  const char* src;
  uint64_t policy;
  int32_t chunk, nchunks;
  uint32_t issued;
  uint32_t pad_;
};

struct StreamShared {
  float4 ring[kStages][kChunkFloats / 4];
  uint32_t cand_key[kCap];
  int32_t cand_j[kCap];
  SelectShared sel;
  uint64_t full[kStages];
  ProducerState prod;
  uint32_t wt[2][kWarps];  // per-warp packed counts of the current tile
  uint32_t b0;             // running threshold: level-1 bin, only rises
  uint32_t top;            // highest level-1 bin holding a candidate
};

// The producer (thread 0) walks the same sequence of chunks the consumers do:
// the rows of this CTA (cluster) in order, rows with a window of at most k
// elements skipped, each row part cut into kChunkBytes pieces from its
// 16-byte aligned start.
__device__ __forceinline__ void producer_start(ProducerState& P, int64_t first_row, int32_t ncl) {
  P.row = first_row - ncl;
  P.bytes = 0;
  P.src = nullptr;
  P.chunk = P.nchunks = 0;
  P.issued = 0;
  P.policy = l2_evict_first_policy();
}

template <int CLUSTER>
__device__ __forceinline__ bool producer_advance(ProducerState& P, const Params& p, int32_t ncl,
                                                 uint32_t rank) {
  while (P.chunk >= P.nchunks) {
    P.row += ncl;
    if (P.row >= p.num_rows) return false;
    const Row r = load_row(p, (int32_t)P.row);
    P.chunk = P.nchunks = 0;
    if (row_is_whole(r, p.k)) continue;
    const Part part = part_of(r, rank, CLUSTER);
    P.bytes = (part.q1 - part.q0) * 16;
    P.src = reinterpret_cast<const char*>(r.base4 + part.q0);
    P.nchunks = (int32_t)((P.bytes + kChunkBytes - 1) / kChunkBytes);
  }
  return true;
}

// Issues the next chunk of the sequence into `slot` (which is issued % kStages).
template <int CLUSTER>
__device__ __noinline__ void producer_issue(StreamShared& S, const Params& p, int32_t ncl, uint32_t rank,
                                            uint32_t slot) {
  ProducerState& P = S.prod;
  fence_proxy_async_smem();  // consumers' reads of the slot precede the async-proxy write
  if (!producer_advance<CLUSTER>(P, p, ncl, rank)) return;
  const int64_t off = (int64_t)P.chunk * kChunkBytes;
  const uint32_t nb = (uint32_t)min((int64_t)kChunkBytes, P.bytes - off);
  mbar_arrive_expect_tx(&S.full[slot], nb);
  bulk_copy_g2s(&S.ring[slot][0], P.src + off, nb, &S.full[slot], P.policy);
  ++P.chunk;
  ++P.issued;
}

// Raises the running threshold: the highest bin b >= b0 such that the list
// holds at least k candidates in bins >= b.  One warp, top-down over the bins
// between the highest candidate bin and b0.  Counts read while other warps
// still add to them can only be low, so the bin found never overshoots.
__device__ __forceinline__ void warp_raise_threshold(StreamShared& S, uint32_t k) {
  const int lane = threadIdx.x & 31;
  // one value for the whole warp, so the loop below stays warp-uniform
  const int b0 = __shfl_sync(0xFFFFFFFFu, (int)*reinterpret_cast<volatile uint32_t*>(&S.b0), 0);
  const int top = __shfl_sync(0xFFFFFFFFu, (int)*reinterpret_cast<volatile uint32_t*>(&S.top), 0);
  uint32_t acc = 0;
  for (int base = top; base >= b0; base -= 32) {
    const int b = base - lane;
    const uint32_t h = b >= b0 ? *reinterpret_cast<volatile uint32_t*>(&S.sel.hist1[b]) : 0u;
    const uint32_t cum = warp_incl_scan(h) + acc;
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, cum >= k);
    if (hit) {
      const int nb = base - (__ffs(hit) - 1);
      if (lane == 0 && nb > b0) atomicMax(&S.b0, (uint32_t)nb);
      return;
    }
    acc = __shfl_sync(0xFFFFFFFFu, cum, 31);
  }
}

__device__ __forceinline__ uint32_t warp_max(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}

// Element e (0..7) of thread t in a tile: sub-tile e/4 covers tile elements
// [0, 2048) or [2048, 4096); thread t holds 4 consecutive ones in each.
__device__ __forceinline__ int32_t tile_offset(int e) {
  return (e < 4 ? 0 : kThreads * 4) + (int)threadIdx.x * 4 + (e & 3);
}

// Writes the flagged elements of the tile at list positions count + their
// ordered rank (sub-tile 0 before sub-tile 1, threads in order).  `ex` is the
// exclusive packed prefix of this thread, `total` the tile's packed total.
__device__ __forceinline__ void write_flagged(StreamShared& S, uint32_t fl, const float x[8],
                                              int32_t tj0, uint32_t count, uint32_t ex,
                                              uint32_t total) {
  uint32_t pos0 = count + (ex & 0xFFFFu);
  uint32_t pos1 = count + (total & 0xFFFFu) + (ex >> 16);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (fl & (1u << e)) {
      const uint32_t pos = e < 4 ? pos0++ : pos1++;
      S.cand_key[pos] = key_of(x[e]);
      S.cand_j[pos] = tj0 + tile_offset(e);
    }
  }
}

// The list is full: raise the threshold with the current tile already counted
// in the histogram, and drop the listed candidates below it (order kept).
// Returns the new list length and the new threshold key in *K0.
__device__ __noinline__ uint32_t compact_list(StreamShared& S, uint32_t count, uint32_t k,
                                              ScanParity& par, uint32_t* K0_out) {
  if ((threadIdx.x >> 5) == 0) warp_raise_threshold(S, k);
  __syncthreads();
  const uint32_t K0 = S.b0 << kShift1;
  const int tid = threadIdx.x;
  uint32_t kept = 0;
  for (uint32_t base = 0; base < count; base += kThreads * 4) {
    const uint32_t e0 = base + tid * 4;
    uint32_t kk[4];
    int32_t jj[4];
    uint32_t keep = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool in = e0 + e < count;
      kk[e] = in ? S.cand_key[e0 + e] : 0u;
      jj[e] = in ? S.cand_j[e0 + e] : 0;
      if (in && kk[e] >= K0) keep |= 1u << e;
    }
    uint32_t tot;
    uint32_t pos = kept + block_excl_scan(__popc(keep), par.next(S.sel), tot);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (keep & (1u << e)) {
        S.cand_key[pos] = kk[e];
        S.cand_j[pos] = jj[e];
        ++pos;
      }
    }
    kept += tot;
  }
  *K0_out = K0;
  return kept;
}

// Selection on the candidate list and ordered emission (the usual end of a row).
template <int CLUSTER>
__device__ __noinline__ void finish_from_list(const Params& p, int64_t row, const int32_t* page_row,
                                              StreamShared& S, uint32_t count, ScanParity& par) {
  const CandSrc src{S.cand_key, S.cand_j, (int32_t)(count < (uint32_t)kCap ? count : (uint32_t)kCap)};
  const Selection sel = select_levels<CLUSTER>(S.sel, src, (uint32_t)p.k, par);
  emit_selected(src, sel, p.out + row * p.k, (uint32_t)p.k, page_row, p.page_bits, S.sel, par);
}

// A row whose candidates did not fit: every pass from global memory.
template <int CLUSTER>
__device__ __noinline__ void finish_from_global(const Params& p, int64_t row, const Row& r,
                                                const Part& part, SelectShared& S, ScanParity& par) {
  select_from_global<CLUSTER>(p, (int32_t)row, r, part, S, par);
}

template <int CLUSTER>
__global__ void __launch_bounds__(kThreads, 2) topk_stream_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StreamShared& S = *reinterpret_cast<StreamShared*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = CLUSTER > 1 ? cluster_rank() : 0u;
  const int32_t cid = (int32_t)(blockIdx.x / CLUSTER), ncl = (int32_t)(gridDim.x / CLUSTER);
  const uint32_t k = (uint32_t)p.k;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&S.full[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  if constexpr (CLUSTER > 1) cluster_sync_all();

  if (tid == 0) {
    producer_start(S.prod, cid, ncl);
    for (uint32_t s = 0; s < (uint32_t)kStages; ++s) producer_issue<CLUSTER>(S, p, ncl, rank, s);
  }

  ScanParity par;
  uint32_t g = 0, wtpar = 0;
  bool timed_out = false;

  for (int64_t row = cid; row < p.num_rows; row += ncl) {
    const Row r = load_row(p, (int32_t)row);
    if (row_is_whole(r, p.k)) {
      emit_whole_window(p, (int32_t)row, r, rank, (uint32_t)CLUSTER);
      continue;
    }
    const Part part = part_of(r, rank, (uint32_t)CLUSTER);
    const int64_t bytes = (part.q1 - part.q0) * 16;
    const int32_t nchunks = (int32_t)((bytes + kChunkBytes - 1) / kChunkBytes);

    for (int b = tid; b < kBins1; b += kThreads) S.sel.hist1[b] = 0u;
    if (tid == 0) {
      S.b0 = 0u;
      S.top = 0u;
    }
    __syncthreads();
    uint32_t count = 0;
    bool overflow = false;

    for (int32_t c = 0; c < nchunks; ++c) {
      const uint32_t slot = g % kStages, parity = (g / kStages) & 1u;
      ++g;
      // After one wait has given up, wait no more: the kernel only finishes its
      // control flow (results unspecified, diagnostic bit set).
      if (!timed_out && !mbar_wait_bounded(&S.full[slot], parity)) timed_out = true;
      const int32_t tj0 = (int32_t)((part.q0 + (int64_t)c * (kChunkFloats / 4)) * 4 - r.head);

      if (overflow) {  // the row already goes to the fallback: only keep the ring moving
        __syncthreads();
        if (tid == 0) producer_issue<CLUSTER>(S, p, ncl, rank, slot);
        continue;
      }

      const float4 va = S.ring[slot][tid], vb = S.ring[slot][kThreads + tid];
      const float x[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
      uint32_t validm = 0xFFu;
      if (!(tj0 >= part.lo && tj0 + kChunkFloats <= part.hi)) {
        validm = 0u;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int32_t j = tj0 + tile_offset(e);
          if (j >= part.lo && j < part.hi) validm |= 1u << e;
        }
      }

      if (c == 0) {
        // First tile of the row: histogram every element, pick the bin of the
        // k-th largest among them, keep only what reaches that bin.
        uint32_t maxbin = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (validm & (1u << e)) {
            const uint32_t bin = key_of(x[e]) >> kShift1;
            atomicAdd(&S.sel.hist1[bin], 1u);
            maxbin = max(maxbin, bin);
          }
        }
        const uint32_t mb = warp_max(maxbin);
        if (lane == 0 && mb > 0) atomicMax(&S.top, mb);
        __syncthreads();
        if (tid == 0) producer_issue<CLUSTER>(S, p, ncl, rank, slot);
        const int32_t nvalid = max(0, min(part.hi, tj0 + kChunkFloats) - max(part.lo, tj0));
        uint32_t b0 = 0;
        if ((uint32_t)nvalid >= k) {
          const Pick pk = block_pick<kBins1, 1>(S.sel.hist1, k, par.next(S.sel), par.next_pick(S.sel));
          b0 = pk.bin;
          if (tid == 0) S.b0 = b0;
        }
        const uint32_t K0 = b0 << kShift1;
        uint32_t fl = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if ((validm & (1u << e)) && key_of(x[e]) >= K0) fl |= 1u << e;
        const uint32_t packed = __popc(fl & 0xFu) | ((uint32_t)__popc(fl >> 4) << 16);
        uint32_t total;
        const uint32_t ex = block_excl_scan(packed, par.next(S.sel), total);
        write_flagged(S, fl, x, tj0, 0u, ex, total);
        count = (total & 0xFFFFu) + (total >> 16);
        continue;
      }

      const float th = edge_float(*reinterpret_cast<volatile uint32_t*>(&S.b0));
      uint32_t fl = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (x[e] >= th) fl |= 1u << e;
      fl &= validm;
      const uint32_t packed = __popc(fl & 0xFu) | ((uint32_t)__popc(fl >> 4) << 16);
      uint32_t maxbin = 0;
      if (fl) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          if (fl & (1u << e)) {
            const uint32_t bin = key_of(x[e]) >> kShift1;
            atomicAdd(&S.sel.hist1[bin], 1u);
            maxbin = max(maxbin, bin);
          }
        }
      }
      const uint32_t incl = warp_incl_scan(packed);
      uint32_t* wt = S.wt[wtpar];
      wtpar ^= 1u;
      if (lane == 31) wt[warp] = incl;
      const uint32_t mb = warp_max(maxbin);
      if (lane == 0 && mb > 0) atomicMax(&S.top, mb);
      __syncthreads();
      if (tid == 0) producer_issue<CLUSTER>(S, p, ncl, rank, slot);
      const uint32_t w = lane < kWarps ? wt[lane] : 0u;
      const uint32_t wincl = warp_incl_scan(w);
      const uint32_t wbase = __shfl_sync(0xFFFFFFFFu, wincl - w, warp);
      const uint32_t total = __shfl_sync(0xFFFFFFFFu, wincl, kWarps - 1);
      const uint32_t tcount = (total & 0xFFFFu) + (total >> 16);

      if (count + tcount <= (uint32_t)kCap) {
        write_flagged(S, fl, x, tj0, count, wbase + incl - packed, total);
        count += tcount;
        if (warp == (c & (kWarps - 1))) warp_raise_threshold(S, k);
        continue;
      }

      // The list is full: raise the threshold with this tile counted, drop the
      // listed candidates below it (order kept), then add the tile's survivors.
      uint32_t K0;
      const uint32_t kept = compact_list(S, count, k, par, &K0);
      uint32_t fl2 = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if ((fl & (1u << e)) && key_of(x[e]) >= K0) fl2 |= 1u << e;
      uint32_t total2;
      const uint32_t ex2 = block_excl_scan(__popc(fl2 & 0xFu) | ((uint32_t)__popc(fl2 >> 4) << 16),
                                           par.next(S.sel), total2);
      const uint32_t t2 = (total2 & 0xFFFFu) + (total2 >> 16);
      if (kept + t2 <= (uint32_t)kCap) {
        write_flagged(S, fl2, x, tj0, kept, ex2, total2);
        count = kept + t2;
      } else {
        overflow = true;
        count = kept;
      }
    }

    // ---- end of the row's stream: select on the list (or fall back) ----
    __syncthreads();
    bool any_over = overflow;
    if constexpr (CLUSTER > 1) {
      if (tid == 0) S.sel.pub_overflow = overflow ? 1u : 0u;
      cluster_sync_all();
      const uint32_t a = smem_addr(&S.sel.pub_overflow);
      uint32_t o = 0;
      for (uint32_t c = 0; c < (uint32_t)CLUSTER; ++c) o |= ld_cluster_u32(peer_addr(a, c));
      any_over = o != 0u;
    }
    if (any_over)
      finish_from_global<CLUSTER>(p, row, r, part, S.sel, par);
    else
      finish_from_list<CLUSTER>(p, row, r.page_row, S, count, par);
  }

  // Every issued chunk was waited for, so nothing is in flight -- unless a
  // wait gave up; then wait (bounded) for the copies still outstanding.
  if (__syncthreads_or(timed_out ? 1 : 0)) {
    if (tid == 0) {
      atomicOr(&g_device_flags, kFlagStreamWaitTimeout);
      const uint32_t issued = S.prod.issued;
      for (uint32_t n = (issued > (uint32_t)kStages ? issued - kStages : 0u); n < issued; ++n)
        mbar_wait_bounded(&S.full[n % kStages], (n / kStages) & 1u);
    }
    __syncthreads();
  }
  if constexpr (CLUSTER > 1) cluster_sync_all();  // peers may still read this CTA's shared memory
}

}  // namespace topk
