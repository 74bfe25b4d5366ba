// Register-resident kernel for short windows (decode-like batches) of the
// packed top-k + page transform (sm_103a).
//
// The operation is the one of topk_pipe.cuh (page "[sglang] [AMD ROCm] GLM-5.x
// Prefill 성능을 66% 끌어올린 Top-K 커널 최적화 분석", sglang PR #37889, Intro
// and sections 1-2; the page's intro names the paged decode kernel this one
// stands beside).  A decode step has few rows of a few thousand keys each,
// so the time is latency, not bandwidth: one CTA of 1024 threads takes a row,
// reads its window from HBM once into registers (16-byte loads from the start
// rounded down to 16 bytes, lanes outside the window masked), and runs the
// exact radix select of topk_device.cuh (12-, 10- and 10-bit digits with an
// early exit) on the registers: each level is one pass of shared-memory
// atomics and one block-wide bucket pick.  The emission keeps, in ascending
// window index, the keys above the k-th largest and the first `quota` equal
// to it, at positions from block-wide prefix counts, through the page
// transform.
//
// Thread t holds quads u * 1024 + t (u < QPT) of the row, so the u-th quads of
// all threads are one contiguous run of the window: walking u outermost and
// threads in order visits the window in ascending index.
#pragma once

#include "topk_device.cuh"

namespace topk {
namespace decode {

constexpr int kThreads = 1024;

// Largest row_stride the kernel with QPT quads a thread serves: every window
// (at most row_stride elements) plus its head (at most 3) fits.
template <int QPT>
constexpr int64_t max_stride() {
  return (int64_t)kThreads * QPT * 4 - 3;
}

// A row's window in registers, as a source of (key, window index) pairs for
// select_levels.
template <int QPT>
struct RegSrc {
  uint32_t key[QPT][4];
  int32_t jq;  // window index of element 0 of the thread's quad 0
  int32_t L;

  __device__ __forceinline__ int32_t index(int u, int e) const { return jq + u * kThreads * 4 + e; }
  __device__ __forceinline__ bool valid(int u, int e) const {
    const int32_t j = index(u, e);
    return j >= 0 && j < L;
  }

  __device__ __forceinline__ void load(const Row& r) {
    const int64_t nq = ((int64_t)r.L + r.head + 3) >> 2;
    L = r.L;
    jq = (int32_t)threadIdx.x * 4 - r.head;
    float4 v[QPT];
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      const int64_t q = (int64_t)u * kThreads + threadIdx.x;
      v[u] = q < nq ? load_window_quad(r, q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < QPT; ++u) {
      key[u][0] = key_of(v[u].x);
      key[u][1] = key_of(v[u].y);
      key[u][2] = key_of(v[u].z);
      key[u][3] = key_of(v[u].w);
    }
  }

  // hist[(key >> shift) & nbins_mask] += 1 for every window element whose key
  // matches prefix T under mask M.
  __device__ __forceinline__ void histogram(uint32_t* hist, uint32_t M, uint32_t T, int shift,
                                            uint32_t nbins_mask) const {
#pragma unroll
    for (int u = 0; u < QPT; ++u)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (valid(u, e) && (key[u][e] & M) == T) atomicAdd(hist + ((key[u][e] >> shift) & nbins_mask), 1u);
  }
};

// Writes the selected window indices of the row, in ascending order, through
// the page transform: per quad tile u, one block-wide scan of the threads'
// counts of keys above the prefix (gt) and equal to it (eq, taken while the
// tie quota lasts).
template <int QPT>
__device__ __forceinline__ void emit(const RegSrc<QPT>& src, const Selection& sel, int32_t* out_row, uint32_t k,
                                     const int32_t* page_row, int32_t page_bits, SelectShared& S, ScanParity& par) {
  uint32_t gt_run = 0, eq_run = 0;
#pragma unroll
  for (int u = 0; u < QPT; ++u) {
    bool is_gt[4], is_eq[4];
    uint32_t ngt = 0, neq = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const bool v = src.valid(u, e);
      const uint32_t pk = src.key[u][e] & sel.M;
      is_gt[e] = v && pk > sel.T;
      is_eq[e] = v && pk == sel.T;
      ngt += is_gt[e];
      neq += is_eq[e];
    }
    uint32_t total;  // 16-bit fields: at most 4 * kThreads = 4096 of each per tile
    const uint32_t ex = block_excl_scan<kThreads>(ngt | (neq << 16), par.next(S), total);
    uint32_t g = gt_run + (ex & 0xFFFFu), q = eq_run + (ex >> 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (is_gt[e] || (is_eq[e] && q < sel.quota)) {
        const uint32_t pos = g + (q < sel.quota ? q : sel.quota);
        if (pos < k)
          out_row[pos] = page_slot(page_row, page_bits, src.index(u, e), src.L);
        else
          atomicOr(&g_device_flags, kFlagBadOutputPosition);  // never expected
      }
      g += is_gt[e];
      q += is_eq[e];
    }
    gt_run += total & 0xFFFFu;
    eq_run += total >> 16;
  }
}

template <int QPT>
__global__ void __launch_bounds__(kThreads, 1) topk_decode_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SelectShared& S = *reinterpret_cast<SelectShared*>(smem_raw);
  ScanParity par;
  wait_for_producer();
  allow_dependents();
  for (int64_t row = blockIdx.x; row < p.num_rows; row += gridDim.x) {
    const Row r = load_row(p, (int32_t)row);
    if (r.L <= p.k) {
      emit_whole_window<kThreads>(p, (int32_t)row, r, 0u, 1u);
      continue;
    }
    RegSrc<QPT> src;
    src.load(r);
    for (int b = threadIdx.x; b < kBins1; b += kThreads) S.hist1[b] = 0u;
    __syncthreads();  // also: every thread is done with the previous row's state
    src.histogram(S.hist1, 0u, 0u, kShift1, kBins1 - 1);
    __syncthreads();
    const Selection sel = select_levels<1, kThreads>(S, src, (uint32_t)p.k, par);
    emit<QPT>(src, sel, p.out + row * p.k, (uint32_t)p.k, r.page_row, p.page_bits, S, par);
  }
}

}  // namespace decode
}  // namespace topk
