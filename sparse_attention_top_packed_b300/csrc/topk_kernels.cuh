// Kernels of the packed top-k + page transform (sm_103a).
//
//   topk_multipass_kernel  one CTA per row (grid-strided): a 12-bit histogram
//                          of the whole window, then 10-bit refinement levels
//                          on the keys that share the chosen prefix, then the
//                          ordered emission -- every pass straight from global
//                          memory.  Simple and always exact.
//   topk_stream_kernel     persistent CTAs (one per SM), or clusters of CTAs
//                          sharing a row, that read every window once from HBM.
//                          Each of the 32 warps owns a contiguous slice of the
//                          row and streams it through its own ring of TMA bulk
//                          copies into shared memory, with no block-wide
//                          synchronisation while streaming.  A running lower
//                          bound on the k-th largest key (first from a sample
//                          of the whole row, then a level-1 histogram bin edge
//                          that only rises, shared by all warps and raised
//                          lock-free) drops almost every element at one
//                          compare; the few that pass are appended, in window
//                          order, to the warp's list in shared memory.  Since
//                          slices are contiguous and in warp order, the lists
//                          concatenated in warp order are in window order.  The
//                          radix select then runs on the lists.  A row whose
//                          candidates overflow a list, or that listed fewer
//                          than k, falls back to the multipass procedure for
//                          that row.
#pragma once

#include "topk_device.cuh"

namespace topk {

__device__ __forceinline__ bool row_is_whole(const Row& r, int32_t k) { return r.L <= k; }

// ---------------------------------------------------------------------------
// Multipass kernel.
// ---------------------------------------------------------------------------
constexpr int kMultipassThreads = 512;

__global__ void __launch_bounds__(kMultipassThreads, 2) topk_multipass_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SelectShared& S = *reinterpret_cast<SelectShared*>(smem_raw);
  ScanParity par;
  wait_for_producer();
  allow_dependents();
  for (int64_t row = blockIdx.x; row < p.num_rows; row += gridDim.x) {
    const Row r = load_row(p, (int32_t)row);
    if (row_is_whole(r, p.k)) {
      emit_whole_window<kMultipassThreads>(p, (int32_t)row, r, 0u, 1u);
      continue;
    }
    const Part part = part_of(r, 0u, 1u);
    select_from_global<1, kMultipassThreads>(p, (int32_t)row, r, part, S, par);
  }
}

// ---------------------------------------------------------------------------
// Streaming kernel.
// ---------------------------------------------------------------------------
constexpr int kStreamThreads = 1024;
constexpr int kStreamWarps = kStreamThreads / 32;
constexpr int kChunkBytes = 2048;              // one warp chunk: 16 floats per lane
constexpr int kChunkQuads = kChunkBytes / 16;  // 128
constexpr int kStages = 2;                     // chunks in flight per warp
constexpr int kWarpCap = 128;                  // list entries per warp (4096 per CTA)

// The producer of one warp (its lane 0): where the next chunk comes from.
struct WarpProducer {
  const char* src;  // next chunk of the current slice
  int64_t left;     // bytes of the slice not yet issued
  int64_t row;      // row of the current slice
  uint32_t issued;  // chunks issued so far
  uint32_t pad_;
  const char* wbeg;  // checked build: the row's window rounded out to 16 bytes
  const char* wend;
};

struct StreamShared {
  float4 ring[kStreamWarps][kStages][kChunkQuads];
  uint32_t list_key[kStreamWarps][kWarpCap];
  int32_t list_j[kStreamWarps][kWarpCap];
  SelectShared sel;
  uint64_t full[kStreamWarps][kStages];
  WarpProducer prod[kStreamWarps];
  uint32_t count[kStreamWarps];  // list lengths at the end of the row
  uint32_t wgt[kStreamWarps];    // per-warp counts for the emission
  uint32_t weq[kStreamWarps];
  uint32_t b0;        // running threshold: level-1 bin, only rises
  uint32_t top;       // highest level-1 bin holding a candidate (may lag)
  uint32_t overflow;  // a list of this row overflowed
};

// Slice of a row part owned by warp w: quads [q0, q1), window indices [lo, hi).
struct Slice {
  int64_t q0, q1;
  int32_t lo, hi;
};

__device__ __forceinline__ Slice slice_of(const Row& r, const Part& part, int w) {
  const int64_t nq = part.q1 - part.q0;
  const int64_t per = (nq + kStreamWarps - 1) / kStreamWarps;
  Slice s;
  s.q0 = min(part.q0 + (int64_t)w * per, part.q1);
  s.q1 = min(s.q0 + per, part.q1);
  s.lo = (int32_t)min(max(s.q0 * 4 - r.head, (int64_t)0), (int64_t)r.L);
  s.hi = (int32_t)min(max(s.q1 * 4 - r.head, (int64_t)0), (int64_t)r.L);
  return s;
}

// Moves the producer of warp w to the next row (of this CTA / cluster) in
// which warp w owns a non-empty slice.
template <int CLUSTER>
__device__ __noinline__ void producer_next_row(WarpProducer& P, const Params& p, int32_t ncl,
                                               uint32_t rank, int w) {
  while (true) {
    P.row += ncl;
    if (P.row >= p.num_rows) {
      P.left = 0;
      return;
    }
    const Row r = load_row(p, (int32_t)P.row);
    if (row_is_whole(r, p.k)) continue;
    const Slice sl = slice_of(r, part_of(r, rank, CLUSTER), w);
    if (sl.q1 > sl.q0) {
      P.src = reinterpret_cast<const char*>(r.base4 + sl.q0);
      P.left = (sl.q1 - sl.q0) * 16;
      if constexpr (kChecked) {
        P.wbeg = reinterpret_cast<const char*>(r.base4);
        P.wend = P.wbeg + (((int64_t)r.L + r.head + 3) >> 2) * 16;
      }
      return;
    }
  }
}

// Lane 0 of warp w: issues the next chunk of the warp's sequence into `slot`
// (= issued % kStages).  The sequence is the slices of the rows in the order
// the warp consumes them, each cut into kChunkBytes pieces.
template <int CLUSTER>
__device__ __forceinline__ void producer_issue(StreamShared& S, const Params& p, int32_t ncl,
                                               uint32_t rank, int w, uint32_t slot, uint64_t policy) {
  WarpProducer& P = S.prod[w];
  if (P.left == 0) {
    if (P.row >= p.num_rows) return;
    producer_next_row<CLUSTER>(P, p, ncl, rank, w);
    if (P.left == 0) return;
  }
  const uint32_t nb = (uint32_t)min((int64_t)kChunkBytes, P.left);
  fence_proxy_async_smem();  // the warp's reads of the slot precede the async-proxy write
  if (!in_bounds(P.src >= P.wbeg && P.src + nb <= P.wend, kSiteWindowCopy)) {
    mbar_arrive(&S.full[w][slot]);  // checked build: the phase completes without the copy
  } else {
    mbar_arrive_expect_tx(&S.full[w][slot], nb);
    bulk_copy_g2s(&S.ring[w][slot][0], P.src, nb, &S.full[w][slot], policy);
  }
  P.src += nb;
  P.left -= nb;
  ++P.issued;
}

// Raises the running threshold (one warp, lock-free): the highest bin b >= b0
// such that at least k elements counted so far lie in bins >= b.  Counts read
// while other warps still add to them can only be low, so the bin found never
// overshoots the k-th largest key.  Also publishes this warp's highest bin.
__device__ __forceinline__ void warp_raise_threshold(StreamShared& S, uint32_t k, uint32_t mbin) {
  const int lane = threadIdx.x & 31;
  const uint32_t mb = warp_max(mbin);
  if (lane == 0) atomicMax(&S.top, mb);
  __syncwarp();
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

// Appends the lane's flagged elements (bit e of m = element e of the lane's 16
// in the slot, element order) at list positions pos, pos+1, ... in ascending e.
// With COUNT, each one is also counted in the level-1 histogram.
template <bool COUNT>
__device__ __forceinline__ void append_flagged(StreamShared& S, int w, const float* xs, uint32_t m,
                                               uint32_t pos, int32_t jb, uint32_t& mbin) {
  while (m) {
    const int e = __ffs(m) - 1;
    m &= m - 1;
    const uint32_t key = key_of(xs[e]);
    if (COUNT) {
      const uint32_t bin = key >> kShift1;
      atomicAdd(&S.sel.hist1[bin], 1u);
      mbin = max(mbin, bin);
    }
    if (in_bounds(pos < (uint32_t)kWarpCap, kSiteCandidate)) {
      S.list_key[w][pos] = key;
      S.list_j[w][pos] = jb + e;
    }
    ++pos;
  }
}

// The warp's list is full: raise the threshold, drop the listed candidates
// below it (order kept).  Returns the new length and the threshold bin.
__device__ __noinline__ uint32_t compact_warp_list(StreamShared& S, int w, uint32_t count, uint32_t k,
                                                   uint32_t mbin, uint32_t* b0_out) {
  const int lane = threadIdx.x & 31;
  warp_raise_threshold(S, k, mbin);
  const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, *reinterpret_cast<volatile uint32_t*>(&S.b0), 0);
  const uint32_t K0 = b0 << kShift1;
  uint32_t kept = 0;
  for (uint32_t i0 = 0; i0 < count; i0 += 32) {
    const uint32_t i = i0 + lane;
    const bool in = i < count;
    const uint32_t key = in ? S.list_key[w][i] : 0u;
    const int32_t j = in ? S.list_j[w][i] : 0;
    const bool keep = in && key >= K0;
    const uint32_t b = __ballot_sync(0xFFFFFFFFu, keep);
    const uint32_t dst = kept + __popc(b & lanemask_lt());
    __syncwarp();
    if (keep) {
      S.list_key[w][dst] = key;
      S.list_j[w][dst] = j;
    }
    kept += __popc(b);
    __syncwarp();
  }
  *b0_out = b0;
  return kept;
}

// Bits of the lane's 16 elements (element order) whose window index jb+e lies
// in [lo, hi).
__device__ __forceinline__ uint32_t valid16(int32_t jb, int32_t lo, int32_t hi) {
  uint32_t m = 0;
#pragma unroll
  for (int e = 0; e < 16; ++e) m |= ((jb + e >= lo && jb + e < hi) ? 1u : 0u) << e;
  return m;
}

// A lane's 16 elements are the 4 consecutive quads 4*lane .. 4*lane+3 of the
// chunk.  They are read in the rotated order q -> quad 4*lane + ((q + lane/2) & 3)
// so that the 8 lanes of each shared-memory phase hit 8 different 16-byte bank
// groups; x[4q+v] therefore holds element 4*((q + lane/2) & 3) + v.  Masks are
// computed in that "rotated" order and turned into element order by a rotate.
__device__ __forceinline__ void load16_rotated(const StreamShared& S, int w, uint32_t slot, int lane,
                                               float x[16]) {
  const int s = (lane >> 1) & 3;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 v = S.ring[w][slot][lane * 4 + ((q + s) & 3)];
    x[4 * q] = v.x;
    x[4 * q + 1] = v.y;
    x[4 * q + 2] = v.z;
    x[4 * q + 3] = v.w;
  }
}

__device__ __forceinline__ uint32_t rotated_to_element_order(uint32_t m, int lane) {
  const uint32_t s4 = 4u * ((lane >> 1) & 3);
  return ((m << s4) | (m >> (16u - s4))) & 0xFFFFu;
}

__device__ __forceinline__ uint32_t element_to_rotated_order(uint32_t m, int lane) {
  const uint32_t s4 = 4u * ((lane >> 1) & 3);
  return ((m >> s4) | (m << (16u - s4))) & 0xFFFFu;
}

// Flags (rotated order) of a lane's 16 elements: bit i set when x[i] >= th.
__device__ __forceinline__ uint32_t flags16(const float x[16], float th) {
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) m |= (x[i] >= th ? 1u : 0u) << i;
  return m;
}

// Histogram of a source made of the warps' lists (refinement levels).
struct ListSrc {
  const StreamShared* S;
  __device__ __forceinline__ void histogram(uint32_t* hist, uint32_t M, uint32_t T, int shift,
                                            uint32_t nbins_mask) const {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t n = S->count[w];
    for (uint32_t i = lane; i < n; i += 32) {
      const uint32_t key = S->list_key[w][i];
      if ((key & M) == T) atomicAdd(hist + ((key >> shift) & nbins_mask), 1u);
    }
  }
};

// Ordered emission from the lists: warp w's selected entries follow those of
// warps 0..w-1 (their slices precede w's in the window).
__device__ __forceinline__ void emit_from_lists(StreamShared& S, const Selection& sel, int32_t* out_row, int32_t L,
                                                uint32_t k_row, const int32_t* page_row,
                                                int32_t page_bits) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t n = S.count[w];
  uint32_t ngt = 0, neq = 0;
  for (uint32_t i = lane; i < n; i += 32) {
    const uint32_t pk = S.list_key[w][i] & sel.M;
    ngt += pk > sel.T;
    neq += pk == sel.T;
  }
  ngt = warp_sum(ngt);
  neq = warp_sum(neq);
  if (lane == 0) {
    S.wgt[w] = ngt;
    S.weq[w] = neq;
  }
  __syncthreads();
  const uint32_t gv = S.wgt[lane], ev = S.weq[lane];
  const uint32_t gi = warp_incl_scan(gv), ei = warp_incl_scan(ev);
  const uint32_t gt_before = __shfl_sync(0xFFFFFFFFu, gi - gv, w);
  const uint32_t eq_before = __shfl_sync(0xFFFFFFFFu, ei - ev, w);
  const uint32_t lt = lanemask_lt();
  uint32_t g = gt_before, q = eq_before;
  for (uint32_t i0 = 0; i0 < n; i0 += 32) {
    const uint32_t i = i0 + lane;
    const bool in = i < n;
    const uint32_t pk = in ? (S.list_key[w][i] & sel.M) : 0u;
    const bool is_gt = in && pk > sel.T;
    const bool is_eq = in && pk == sel.T;
    const uint32_t bg = __ballot_sync(0xFFFFFFFFu, is_gt), be = __ballot_sync(0xFFFFFFFFu, is_eq);
    const uint32_t gl = g + __popc(bg & lt), ql = q + __popc(be & lt);
    if (is_gt || (is_eq && ql < sel.quota)) {
      const uint32_t pos = sel.off + gl + (ql < sel.quota ? ql : sel.quota);
      if (pos < k_row)
        out_row[pos] = page_slot(page_row, page_bits, S.list_j[w][i], L);
      else
        atomicOr(&g_device_flags, kFlagBadOutputPosition);  // never expected
    }
    g += __popc(bg);
    q += __popc(be);
  }
}

template <int CLUSTER>
__device__ __noinline__ void finish_from_lists(const Params& p, int64_t row, const int32_t* page_row, int32_t L,
                                               StreamShared& S, ScanParity& par) {
  const ListSrc src{&S};
  const Selection sel = select_levels<CLUSTER, kStreamThreads>(S.sel, src, (uint32_t)p.k, par);
  emit_from_lists(S, sel, p.out + row * p.k, L, (uint32_t)p.k, page_row, p.page_bits);
}

template <int CLUSTER>
__device__ __noinline__ void finish_from_global(const Params& p, int64_t row, const Row& r,
                                                const Part& part, SelectShared& S, ScanParity& par) {
  select_from_global<CLUSTER, kStreamThreads>(p, (int32_t)row, r, part, S, par);
}

// Whole CTA, entered through a barrier with S.sel.hist1 zero: the 22-bit key
// prefix that about 1.4 k of the row's elements reach, estimated from a sample
// spread evenly over the whole window (every CTA of a cluster computes the
// same): 4096 elements, or 16384 when 4096 would put fewer than ~128 above
// that rank.  Two digits, 12 and 10 bits, the second reading the sample again
// (from L2).  Leaves hist1 zero; ends with a barrier.
__device__ __noinline__ uint32_t stream_sample_threshold(StreamShared& S, const Params& p, const Row& r,
                                                         ScanParity& par) {
  const int tid = threadIdx.x;
  const int64_t nq = ((int64_t)r.L + r.head + 3) >> 2;
  const bool long_sample = (int64_t)r.L * 128 > (int64_t)14 * p.k * 4096 / 10;
  const int64_t nsamp = long_sample ? 16384 : 4096, ns = nsamp / 4;
  auto quad = [&](int64_t s) { return ((2 * s + 1) * nq) / (2 * ns); };
  auto key_at = [&](int64_t q, const float4& v, int e) {
    const int64_t j = q * 4 - r.head + e;
    const float x = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    return (j >= 0 && j < r.L) ? key_of(x) : 0u;  // outside the window: the lowest key
  };
  for (int64_t s = tid; s < ns; s += kStreamThreads) {
    const int64_t q = quad(s);
    const float4 v = load_window_quad(r, q, kSiteSampleLoad);
#pragma unroll
    for (int e = 0; e < 4; ++e) atomicAdd(&S.sel.hist1[key_at(q, v, e) >> kShift1], 1u);
  }
  for (int b = tid; b < kBins23; b += kStreamThreads) S.sel.hist2[b] = 0u;
  __syncthreads();
  const uint32_t R = (uint32_t)min((7 * (int64_t)p.k * nsamp) / (5 * (int64_t)r.L) + 1, nsamp);
  const Pick a = block_pick<kBins1, 1, kStreamThreads>(S.sel.hist1, R, par.next(S.sel), par.next_pick(S.sel));
  for (int64_t s = tid; s < ns; s += kStreamThreads) {
    const int64_t q = quad(s);
    const float4 v = load_window_quad(r, q, kSiteSampleLoad);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t key = key_at(q, v, e);
      if ((key >> kShift1) == a.bin) atomicAdd(&S.sel.hist2[(key >> kShift2) & (kBins23 - 1)], 1u);
    }
  }
  __syncthreads();
  const Pick b = block_pick<kBins23, 1, kStreamThreads>(S.sel.hist2, R - a.above, par.next(S.sel),
                                                        par.next_pick(S.sel));
  for (int i = tid; i < kBins1; i += kStreamThreads) S.sel.hist1[i] = 0u;
  __syncthreads();
  return (a.bin << kShift1) | (b.bin << kShift2);
}

template <int CLUSTER>
__global__ void __launch_bounds__(kStreamThreads, 1) topk_stream_kernel(Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StreamShared& S = *reinterpret_cast<StreamShared*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const uint32_t rank = CLUSTER > 1 ? cluster_rank() : 0u;
  const int32_t cid = (int32_t)(blockIdx.x / CLUSTER), ncl = (int32_t)(gridDim.x / CLUSTER);
  const uint32_t k = (uint32_t)p.k;
  const uint64_t policy = l2_evict_first_policy();
  wait_for_producer();  // the prologue below already reads the inputs
  allow_dependents();

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&S.full[w][s], 1);
    fence_barrier_init();
    WarpProducer& P = S.prod[w];
    P.row = (int64_t)cid - ncl;
    P.left = 0;
    P.src = nullptr;
    P.issued = 0;
    P.wbeg = P.wend = nullptr;
    for (uint32_t s = 0; s < (uint32_t)kStages; ++s) producer_issue<CLUSTER>(S, p, ncl, rank, w, s, policy);
  }
  __syncthreads();
  if constexpr (CLUSTER > 1) cluster_sync_all();

  ScanParity par;
  uint32_t g = 0;  // chunks this warp consumed
  bool timed_out = false;

  for (int64_t row = cid; row < p.num_rows; row += ncl) {
    const Row r = load_row(p, (int32_t)row);
    if (row_is_whole(r, p.k)) {
      emit_whole_window<kStreamThreads>(p, (int32_t)row, r, rank, (uint32_t)CLUSTER);
      continue;
    }
    const Part part = part_of(r, rank, (uint32_t)CLUSTER);
    const Slice sl = slice_of(r, part, w);
    const int32_t nch = (int32_t)(((sl.q1 - sl.q0) * 16 + kChunkBytes - 1) / kChunkBytes);

    for (int b = tid; b < kBins1; b += kStreamThreads) S.sel.hist1[b] = 0u;
    __syncthreads();
    // the row's starting threshold from a sample; it only rises afterwards
    const uint32_t thr = stream_sample_threshold(S, p, r, par);
    const float th0 = key_floor_float(thr);
    if (tid == 0) {
      S.b0 = thr >> kShift1;
      S.top = 0u;
      S.overflow = 0u;
    }
    __syncthreads();

    uint32_t count = 0, mbin = 0;
    bool over = false;

    // ---- the warp's slice: one compare per element against the running
    // threshold; survivors appended in order; no block-wide synchronisation.
    for (int32_t c = 0; c < nch; ++c) {
      const uint32_t slot = g % kStages;
      if (!timed_out && !mbar_wait_bounded(&S.full[w][slot], (g / kStages) & 1u)) timed_out = true;
      ++g;
      float x[16];
      load16_rotated(S, w, slot, lane, x);
      const int32_t jb = (int32_t)((sl.q0 + (int64_t)c * kChunkQuads) * 4 - r.head) + 16 * lane;
      if (!over) {
        const float th = fmaxf(th0, edge_float(*reinterpret_cast<volatile uint32_t*>(&S.b0)));
        uint32_t m = rotated_to_element_order(flags16(x, th), lane);
        if (c == 0 || c == nch - 1) m &= valid16(jb, sl.lo, sl.hi);
        uint32_t cnt = __popc(m);
        uint32_t incl = warp_incl_scan(cnt);
        uint32_t total = __shfl_sync(0xFFFFFFFFu, incl, 31);
        const float* xs = reinterpret_cast<const float*>(&S.ring[w][slot][lane * 4]);
        if (total != 0) {
          if (count + total > (uint32_t)kWarpCap) {
            uint32_t b0;
            count = compact_warp_list(S, w, count, k, mbin, &b0);
            const float th2 = fmaxf(th0, edge_float(b0));
            uint32_t m2 = 0;
            for (uint32_t mm = m; mm; mm &= mm - 1) {
              const int e = __ffs(mm) - 1;
              if (xs[e] >= th2) m2 |= 1u << e;
            }
            m = m2;
            cnt = __popc(m);
            incl = warp_incl_scan(cnt);
            total = __shfl_sync(0xFFFFFFFFu, incl, 31);
            if (count + total > (uint32_t)kWarpCap) {
              over = true;
              if (lane == 0) S.overflow = 1u;
            }
          }
          if (!over) {
            append_flagged<true>(S, w, xs, m, count + incl - cnt, jb, mbin);
            count += total;
          }
        }
      }
      __syncwarp();
      if (lane == 0) producer_issue<CLUSTER>(S, p, ncl, rank, w, slot, policy);
      if (!over && (c <= 3 || (c & 3) == 0)) warp_raise_threshold(S, k, mbin);
    }
    if (lane == 0) S.count[w] = over || !in_bounds(count <= (uint32_t)kWarpCap, kSiteRegion) ? 0u : count;

    // ---- end of the row's stream: select on the lists, or fall back when a
    // list overflowed or the sampled threshold left fewer than k candidates
    // in the cluster ----
    __syncthreads();
    uint32_t listed = 0;
    for (int i = 0; i < kStreamWarps; ++i) listed += S.count[i];
    bool any_over = S.overflow != 0u || listed < k;
    if constexpr (CLUSTER > 1) {
      if (tid == 0) {
        S.sel.pub_overflow = S.overflow;
        S.sel.pub_count = listed;
      }
      cluster_sync_all();
      const uint32_t a = smem_addr(&S.sel.pub_overflow), ac = smem_addr(&S.sel.pub_count);
      uint32_t o = 0, n = 0;
      for (uint32_t c = 0; c < (uint32_t)CLUSTER; ++c) {
        o |= ld_cluster_u32(peer_addr(a, c));
        n += ld_cluster_u32(peer_addr(ac, c));
      }
      any_over = o != 0u || n < k;
    }
    if (any_over)
      finish_from_global<CLUSTER>(p, row, r, part, S.sel, par);
    else
      finish_from_lists<CLUSTER>(p, row, r.page_row, r.L, S, par);
  }

  // Every issued chunk was waited for, so nothing is in flight -- unless a
  // wait gave up; then wait (bounded) for the copies still outstanding.
  if (__syncthreads_or(timed_out ? 1 : 0)) {
    if (lane == 0) {
      atomicOr(&g_device_flags, kFlagStreamWaitTimeout);
      const uint32_t issued = S.prod[w].issued;
      for (uint32_t n = (issued > (uint32_t)kStages ? issued - kStages : 0u); n < issued; ++n)
        mbar_wait_bounded(&S.full[w][n % kStages], (n / kStages) & 1u);
    }
    __syncthreads();
  }
  if constexpr (CLUSTER > 1) cluster_sync_all();  // peers may still read this CTA's shared memory
}

}  // namespace topk
