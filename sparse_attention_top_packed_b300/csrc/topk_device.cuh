// Device building blocks of the packed top-k + page transform (sm_103a).
//
// Operation (page "[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66% 끌어올린 Top-K 커널
// 최적화 분석", sglang PR #37889): row i reads the window
//   scores[i * row_stride + row_starts[i] + j], 0 <= j < seq_lens[i]
// (Intro: packed layout; section 1: TopKPackedParams), selects the k largest
// (ties to the lower j), and writes the chosen j in ascending order through the
// page transform of section 1 (get_transform: table row = row_to_batch[i] or i),
// padding with -1.
//
// Selection is an exact radix select on 32-bit order-preserving keys, in three
// digit levels: bits [20,32) (4096 bins), [10,20) and [0,10) (1024 bins each).
// After each level the block knows the key prefix T of the k-th largest element
// under mask M, how many elements lie strictly above it (gt) and how many of the
// prefix-equal elements are still to be taken (r).  A level stops the descent
// early when every prefix-equal element is taken.  The emission then keeps, in
// ascending j, every element with (key & M) > T and the first r with
// (key & M) == T -- the tie rule.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace topk {

constexpr int kMaxWarps = 32;  // largest CTA: 1024 threads

constexpr int kBins1 = 4096;  // level 1: key bits [20, 32)
constexpr int kShift1 = 20;
constexpr int kBins23 = 1024;  // levels 2 and 3: bits [10, 20) and [0, 10)
constexpr int kShift2 = 10;
constexpr int kShift3 = 0;

// Device-side diagnostic bits (see topk_packed_device_flags).
constexpr uint32_t kFlagStreamWaitTimeout = 1u;
constexpr uint32_t kFlagBadOutputPosition = 2u;

// Default bound of a wait inside a kernel: ~2 s.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// The diagnostic word (the library is one translation unit).
__device__ uint32_t g_device_flags;

// ---------------------------------------------------------------------------
// Bounds checks of the checked build (compiled with TOPK_CHECKED).  Every
// global-memory access whose address is computed (window loads and bulk
// copies, page-table reads, descriptor reads) and every shared-memory index
// that is not in range by construction (a bin taken with a mask of the
// table's size is) goes through in_bounds(ok, site).  In the normal build
// that is the constant true and costs nothing.  In the checked build a false
// `ok` sets bit 2 of the diagnostics word, records `site` in bits 8-15 if no
// violation was recorded before, and the caller skips the access (a load
// gives zero).  Nothing traps.
// ---------------------------------------------------------------------------
#ifdef TOPK_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

constexpr uint32_t kFlagOutOfBounds = 4u;
constexpr int kSiteShift = 8;
constexpr uint32_t kSiteMask = 0xFFu << kSiteShift;

// Which check failed first (bits 8-15 of the diagnostics word).
enum CheckSite : uint32_t {
  kSiteRowWindow = 1,   // a row's window leaves its buffer row (a broken precondition: recorded, not skipped)
  kSiteRowIndex = 2,    // a descriptor read for a row outside [0, num_rows)
  kSiteWindowLoad = 3,  // a plain load of quads outside the row's window rounded out to 16 bytes
  kSiteWindowCopy = 4,  // a bulk copy of quads outside the row's window rounded out to 16 bytes
  kSitePageRead = 5,    // a page-table read for a window index outside [0, L)
  kSitePageStage = 6,   // a read of a shared page stage outside the entries staged
  kSiteCandidate = 7,   // a candidate stored outside its region or the positions reserved
  kSiteRegion = 8,      // a region or list count beyond its capacity
  kSiteStaging = 9,     // a staged output position beyond the staging row
  kSiteSampleLoad = 10, // a sample quad outside the window
};

#ifdef TOPK_CHECKED
__device__ __noinline__ void record_violation(uint32_t site) {
  uint32_t cur = *reinterpret_cast<volatile uint32_t*>(&g_device_flags);
  for (int i = 0; i < 64; ++i) {  // bounded: every failed exchange means another thread wrote the word
    uint32_t want = cur | kFlagOutOfBounds;
    if ((cur & kSiteMask) == 0u) want |= (site << kSiteShift) & kSiteMask;
    if (want == cur) return;
    const uint32_t prev = atomicCAS(&g_device_flags, cur, want);
    if (prev == cur) return;
    cur = prev;
  }
  atomicOr(&g_device_flags, kFlagOutOfBounds);
}
#endif

__device__ __forceinline__ bool in_bounds(bool ok, uint32_t site) {
#ifdef TOPK_CHECKED
  if (!ok) record_violation(site);
  return ok;
#else
  (void)ok;
  (void)site;
  return true;
#endif
}

struct Params {
  const float* scores;
  int64_t row_stride;
  const int32_t* seq_lens;
  const int32_t* row_starts;
  const int32_t* row_to_batch;  // may be null: identity
  const int32_t* page_table;
  int64_t pt_stride;
  int32_t page_bits;
  int32_t k;
  int32_t* out;
  int32_t num_rows;
  uint32_t stream_wait_ns;  // bound of a wait for a streamed chunk (0: kWaitLimitNs)
  uint32_t test_flags;      // kTestUnsatisfiedWait: see below
};

// Test switch: each streaming warp first waits, bounded by the stream-chunk
// limit, on an mbarrier that nothing completes, so that the wait runs out and
// the give-up path runs (diagnostic bit 0, rows finished by the exact path,
// outstanding copies drained at exit).
constexpr uint32_t kTestUnsatisfiedWait = 1u;

__device__ __forceinline__ uint64_t stream_wait_limit(const Params& p) {
  return p.stream_wait_ns ? (uint64_t)p.stream_wait_ns : kWaitLimitNs;
}


// ---------------------------------------------------------------------------
// Keys.  key(x) orders like x for every non-NaN float; -0.0 is first turned
// into +0.0 so the two tie (IEEE compares them equal).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t key_of(float x) {
  uint32_t u = __float_as_uint(x);
  u = (u == 0x80000000u) ? 0u : u;
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}

// A float f with, for every non-NaN x:  x >= f  <=>  key(x) >= key.
// The smallest non-NaN key is key(-inf) = 0x007FFFFF; every key at or below
// it maps to -inf (decoding those bit patterns would give a NaN, which no x
// reaches).  Above it the decoded float is exact: key 0x7FFFFFFF (no float
// has it, -0.0 being folded into +0.0) decodes to -0.0, and x >= -0.0 holds
// exactly for the x whose key is at least key(+0.0) = 0x80000000.
__device__ __forceinline__ float key_floor_float(uint32_t key) {
  if (key <= 0x007FFFFFu) return __uint_as_float(0xFF800000u);
  const uint32_t u = (key & 0x80000000u) ? (key ^ 0x80000000u) : ~key;
  return __uint_as_float(u);
}

// The float at the lower edge of level-1 bin b:
//   x >= edge_float(b)  <=>  key(x) >= (b << 20)   for every non-NaN x.
__device__ __forceinline__ float edge_float(uint32_t b) { return key_floor_float(b << kShift1); }

// ---------------------------------------------------------------------------
// Element types of the score buffer (the page's `float* scores`, or a 16-bit
// buffer of the same values).  A 16-byte quad holds kPerQuad elements; decode
// gives their exact values as floats -- every bfloat16 and binary16 value is a
// binary32 value -- so keys, order and ties are those of the same values
// stored as 32-bit floats.  bits_at gives the binary32 pattern of element e of
// a run of elements.
//
// The 16-bit types also compare a 32-bit word of two elements with a
// threshold in one packed instruction: for an element x of the type and any
// float t, x >= t exactly when x >= the smallest value of the type that is at
// least t (t rounded toward +inf), which is what threshold_pair holds in both
// halves; ge_pair gives bit 0 for the low element, bit 1 for the high one.
// ---------------------------------------------------------------------------
struct ElemF32 {
  static constexpr int kPerQuad = 4, kBytes = 4;
  __device__ __forceinline__ static void decode(const float4& q, float (&x)[4]) {
    x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
  }
  __device__ __forceinline__ static uint32_t bits_at(const void* run, int e) {
    return static_cast<const uint32_t*>(run)[e];
  }
};

// bfloat16: the upper half of a binary32 pattern.
struct ElemBF16 {
  static constexpr int kPerQuad = 8, kBytes = 2;
  __device__ __forceinline__ static float value(uint32_t h) { return __uint_as_float(h << 16); }
  __device__ __forceinline__ static void decode(const float4& q, float (&x)[8]) {
    const uint32_t w[4] = {__float_as_uint(q.x), __float_as_uint(q.y), __float_as_uint(q.z), __float_as_uint(q.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);            // element 2i: the low half (little endian)
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  __device__ __forceinline__ static uint32_t bits_at(const void* run, int e) {
    return (uint32_t)static_cast<const uint16_t*>(run)[e] << 16;
  }
  __device__ __forceinline__ static uint32_t threshold_pair(float t) {
    const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_ru(t));
    return h | (h << 16);
  }
  __device__ __forceinline__ static uint32_t ge_pair(uint32_t w, uint32_t t2) {
    const uint32_t m = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&w),
                                   *reinterpret_cast<const __nv_bfloat162*>(&t2));
    return (m & 1u) | ((m >> 15) & 2u);
  }
};

// IEEE binary16, decoded by the CUDA conversion.
struct ElemF16 {
  static constexpr int kPerQuad = 8, kBytes = 2;
  __device__ __forceinline__ static float value(uint32_t h) { return __half2float(__ushort_as_half((unsigned short)h)); }
  __device__ __forceinline__ static void decode(const float4& q, float (&x)[8]) {
    const uint32_t w[4] = {__float_as_uint(q.x), __float_as_uint(q.y), __float_as_uint(q.z), __float_as_uint(q.w)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = value(w[i] & 0xFFFFu);
      x[2 * i + 1] = value(w[i] >> 16);
    }
  }
  __device__ __forceinline__ static uint32_t bits_at(const void* run, int e) {
    return __float_as_uint(value(static_cast<const uint16_t*>(run)[e]));
  }
  __device__ __forceinline__ static uint32_t threshold_pair(float t) {
    const uint32_t h = __half_as_ushort(__float2half_ru(t));
    return h | (h << 16);
  }
  __device__ __forceinline__ static uint32_t ge_pair(uint32_t w, uint32_t t2) {
    const uint32_t m = __hge2_mask(*reinterpret_cast<const __half2*>(&w), *reinterpret_cast<const __half2*>(&t2));
    return (m & 1u) | ((m >> 15) & 2u);
  }
};

// ---------------------------------------------------------------------------
// Row addressing (section 1 and section 2 of the page).  The window start is
// rounded down to a 16-byte boundary of its ABSOLUTE address, so the rounding
// is right for any row_stride; `head` lanes before the window and the lanes
// past its end are masked in registers.  The buffer is never written.
// ---------------------------------------------------------------------------
struct Row {
  int32_t L;                // window length, clamped at 0
  const float4* base4;      // 16-byte aligned, at or before the window start
  int32_t head;             // window index 0 is element `head` of base4[0]
  const int32_t* page_row;  // page_table + table_row * pt_stride; null without a page table
};

// Checked build: the row index of a descriptor read, and the caller's
// precondition 0 <= start, start + L <= row_stride for a row that is read.
__device__ __forceinline__ bool row_index_ok(const Params& p, int64_t row) {
  return in_bounds(row >= 0 && row < p.num_rows, kSiteRowIndex);
}

__device__ __forceinline__ void check_row_window(const Params& p, int32_t L, int32_t start) {
  if constexpr (kChecked)
    if (L > p.k) in_bounds(start >= 0 && (int64_t)start + L <= p.row_stride, kSiteRowWindow);
}

__device__ __forceinline__ Row load_row(const Params& p, int32_t row) {
  Row r;
  int32_t L = 0, start = 0;
  if (row_index_ok(p, row)) {
    L = __ldg(p.seq_lens + row);
    start = __ldg(p.row_starts + row);
  }
  check_row_window(p, L, start);
  r.L = L > 0 ? L : 0;
  const float* w = p.scores + (int64_t)row * p.row_stride + start;
  const uintptr_t a = reinterpret_cast<uintptr_t>(w);
  r.head = (int32_t)((a & 15u) >> 2);
  r.base4 = reinterpret_cast<const float4*>(a & ~(uintptr_t)15u);
  const int64_t table_row = p.row_to_batch && row_index_ok(p, row) ? (int64_t)__ldg(p.row_to_batch + row) : (int64_t)row;
  r.page_row = p.page_table ? p.page_table + table_row * p.pt_stride : nullptr;
  return r;
}

// Checked build: quads [q, q + n) of r.base4 lie inside the row's window
// rounded out to 16 bytes (EPQ elements a quad).
template <int EPQ = 4>
__device__ __forceinline__ bool window_quads_ok(const Row& r, int64_t q, int64_t n, uint32_t site) {
  if constexpr (!kChecked) return true;
  const int64_t nq = ((int64_t)r.L + r.head + EPQ - 1) / EPQ;
  return in_bounds(q >= 0 && n >= 0 && q + n <= nq, site);
}

// A 16-byte window load, zero when the checked build rejects it.
template <int EPQ = 4>
__device__ __forceinline__ float4 load_window_quad(const Row& r, int64_t q, uint32_t site = kSiteWindowLoad) {
  if (!window_quads_ok<EPQ>(r, q, 1, site)) return make_float4(0.f, 0.f, 0.f, 0.f);
  return __ldg(r.base4 + q);
}

// The part of a row one CTA of a cluster owns: quads [q0, q1) of base4, window
// indices [lo, hi).  Parts are contiguous and in rank order.
struct Part {
  int64_t q0, q1;
  int32_t lo, hi;
};

__device__ __forceinline__ Part part_of(const Row& r, uint32_t rank, uint32_t parts) {
  const int64_t nq = ((int64_t)r.L + r.head + 3) >> 2;
  const int64_t per = (nq + parts - 1) / parts;
  Part s;
  s.q0 = min((int64_t)rank * per, nq);
  s.q1 = min(s.q0 + per, nq);
  const int64_t lo = s.q0 * 4 - r.head, hi = s.q1 * 4 - r.head;
  s.lo = (int32_t)max(lo, (int64_t)0);
  s.hi = (int32_t)min(hi, (int64_t)r.L);
  if (s.hi < s.lo) s.hi = s.lo;
  return s;
}

// Section 1's transform: page from the high bits of j, offset from the low
// bits (j a window index of a window of length L).
__device__ __forceinline__ int32_t page_slot(const int32_t* page_row, int32_t page_bits, int32_t j, int32_t L) {
  if (page_row == nullptr) return j;  // no page table: the window index itself
  if (!in_bounds((uint32_t)j < (uint32_t)L, kSitePageRead)) return 0;
  return __ldg(page_row + (j >> page_bits)) * (1 << page_bits) + (j & ((1 << page_bits) - 1));
}

// A window no longer than k: every index is taken; slots past L are -1.
template <int NT>
__device__ __forceinline__ void emit_whole_window(const Params& p, int32_t row, const Row& r,
                                                  uint32_t part, uint32_t parts) {
  int32_t* o = p.out + (int64_t)row * p.k;
  for (int32_t t = (int32_t)(part * NT + threadIdx.x); t < p.k; t += (int32_t)(parts * NT))
    o[t] = t < r.L ? page_slot(r.page_row, p.page_bits, t, r.L) : -1;
}

// ---------------------------------------------------------------------------
// PTX helpers: cluster, distributed shared memory, mbarrier, bulk copy.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory word in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t peer_addr(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
               ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// Plain arrival (release): the caller's earlier shared-memory reads of the
// guarded data are done before the phase can complete.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// try_wait that may suspend the thread (not spin) for up to `ns` nanoseconds
// while the phase is incomplete, so waiting warps leave issue slots free.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\t"
               "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
               "selp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "r"(ns) : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most
// `limit_ns`.  Returns false when it gave up (the caller records a diagnostic
// bit).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  const uint32_t hint = limit_ns < 20000u ? (uint32_t)limit_ns : 20000u;
  while (!mbar_try_wait_sleep(bar, parity, hint)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
    __nanosleep(64);
  }
  return true;
}

// Programmatic dependent launch.  The page's section 2 has the kernel wait for
// the grid that produces the scores (its PDLWaitPrimary) before it touches
// them.  Here every kernel calls wait_for_producer after the part of its
// prologue that reads no input (shared-memory and barrier set-up) and before
// its first read of any argument array; launched with programmatic stream
// serialization it can then start while the previous kernel on the stream
// still runs.  Without that launch attribute the wait returns at once.
// allow_dependents lets the next kernel on the stream start its own prologue;
// that kernel's wait still holds it until this grid has completed.
__device__ __forceinline__ void wait_for_producer() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Streaming warp, before its first chunk: under kTestUnsatisfiedWait, waits
// on `never` (initialised, never arrived on) until the stream-chunk limit runs
// out, and records the give-up.
__device__ __forceinline__ void test_unsatisfied_wait(const Params& p, uint64_t* never, bool& timed_out) {
  if ((p.test_flags & kTestUnsatisfiedWait) && !mbar_wait_bounded(never, 0u, stream_wait_limit(p))) timed_out = true;
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// ---------------------------------------------------------------------------
// Block-wide scans.  Counts travel packed: low 16 bits / high 16 bits, each
// at most 2048 per call, so the fields never carry into each other.
// `scratch` holds NT/32 words; callers alternate two buffers between calls
// (every call contains one __syncthreads, which makes two enough).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xFFFFFFFFu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

__device__ __forceinline__ uint32_t warp_incl_suffix(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_down_sync(0xFFFFFFFFu, v, o);
    if (lane + o < 32) v += n;
  }
  return v;
}

__device__ __forceinline__ uint32_t warp_sum(uint32_t v) { return __reduce_add_sync(0xFFFFFFFFu, v); }

__device__ __forceinline__ uint32_t warp_max(uint32_t v) { return __reduce_max_sync(0xFFFFFFFFu, v); }

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive prefix of v over threads in index order; `total` gets the sum.
template <int NT>
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* scratch, uint32_t& total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t incl = warp_incl_scan(v);
  if (lane == 31) scratch[warp] = incl;
  __syncthreads();
  const uint32_t wt = lane < NW ? scratch[lane] : 0u;
  const uint32_t wincl = warp_incl_scan(wt);
  const uint32_t wexcl = __shfl_sync(0xFFFFFFFFu, wincl - wt, warp);
  total = __shfl_sync(0xFFFFFFFFu, wincl, NW - 1);
  return wexcl + incl - v;
}

template <int NT>
__device__ __forceinline__ uint32_t block_sum(uint32_t v, uint32_t* scratch) {
  uint32_t total;
  block_excl_scan<NT>(v, scratch, total);
  return total;
}

// ---------------------------------------------------------------------------
// Bucket pick: the largest bin b with sum(hist[b..]) >= r, where hist is this
// CTA's histogram, or (CLUSTER > 1) the sum of the histograms at the same
// shared-memory offset in every CTA of the cluster.  Returns, to every thread,
// the bin, `above` = sum(hist[b+1..]) and `count` = hist[b].  The caller
// guarantees sum(hist) >= r >= 1.
// ---------------------------------------------------------------------------
struct Pick {
  uint32_t bin, above, count;
};

template <int NBINS, int CLUSTER, int NT>
__device__ __forceinline__ Pick block_pick(const uint32_t* hist, uint32_t r, uint32_t* scratch,
                                           Pick* slot) {
  constexpr int B = NBINS / NT;  // bins per thread
  constexpr int NW = NT / 32;
  static_assert(B == 1 || B == 2 || B == 4 || B == 8, "bins per thread");
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  uint32_t h[B];
  if constexpr (CLUSTER == 1) {
#pragma unroll
    for (int i = 0; i < B; ++i) h[i] = hist[t * B + i];
  } else {
#pragma unroll
    for (int i = 0; i < B; ++i) h[i] = 0;
    const uint32_t local = smem_addr(hist + t * B);
#pragma unroll
    for (int c = 0; c < CLUSTER; ++c) {
      const uint32_t a = peer_addr(local, (uint32_t)c);
      if constexpr (B >= 4) {
#pragma unroll
        for (int i = 0; i < B; i += 4) {
          const uint4 v = ld_cluster_v4(a + 4u * i);
          h[i] += v.x; h[i + 1] += v.y; h[i + 2] += v.z; h[i + 3] += v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < B; ++i) h[i] += ld_cluster_u32(a + 4u * i);
      }
    }
  }
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < B; ++i) s += h[i];
  // suffix over threads: sum of s over threads > t
  const uint32_t incl = warp_incl_suffix(s);
  if (lane == 0) scratch[warp] = incl;
  if (t == 0) *slot = Pick{0u, 0u, 0u};
  __syncthreads();
  const uint32_t wt = lane < NW ? scratch[lane] : 0u;
  const uint32_t wsuf = warp_incl_suffix(wt);
  const uint32_t above_warps = __shfl_sync(0xFFFFFFFFu, wsuf - wt, warp);
  uint32_t run = above_warps + incl - s;  // sum over bins above this thread's bins
#pragma unroll
  for (int i = B - 1; i >= 0; --i) {
    const uint32_t prev = run;
    run += h[i];
    if (prev < r && run >= r) *slot = Pick{(uint32_t)(t * B + i), prev, h[i]};
  }
  __syncthreads();
  return *slot;
}

// Sum of this CTA's own hist[b] for b > bin (only needed with clusters).
template <int NBINS, int NT>
__device__ __forceinline__ uint32_t own_above(const uint32_t* hist, uint32_t bin, uint32_t* scratch) {
  constexpr int B = NBINS / NT;
  uint32_t s = 0;
#pragma unroll
  for (int i = 0; i < B; ++i) {
    const uint32_t b = threadIdx.x * B + i;
    if (b > bin) s += hist[b];
  }
  return block_sum<NT>(s, scratch);
}

// ---------------------------------------------------------------------------
// A row part read straight from global memory (16-byte loads, masked lanes),
// as a source of (key, j) pairs: for the multipass kernel and for the
// streaming kernel's fallback.  The emission walks it in "tiles" of NT*4
// elements in ascending j, 4 per thread.
// ---------------------------------------------------------------------------
template <int NT>
struct GlobalSrc {
  const float4* base4;
  int64_t q0, q1;
  int32_t head, lo, hi;
  int32_t L;  // the row's window length

  __device__ __forceinline__ float4 load(int64_t q) const {
    if constexpr (kChecked) {
      Row r;
      r.L = L;
      r.base4 = base4;
      r.head = head;
      r.page_row = nullptr;
      return load_window_quad(r, q);
    }
    return __ldg(base4 + q);
  }

  // hist[(key >> shift) & (nbins-1)] += 1 for every element whose key matches
  // prefix T under mask M.
  __device__ __forceinline__ void histogram(uint32_t* hist, uint32_t M, uint32_t T, int shift,
                                            uint32_t nbins_mask) const {
    constexpr int U = 4;
    for (int64_t q = q0 + threadIdx.x; q < q1; q += (int64_t)NT * U) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t qq = q + (int64_t)u * NT;
        v[u] = qq < q1 ? load(qq) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t qq = q + (int64_t)u * NT;
        const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
        const int64_t j0 = qq * 4 - head;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int64_t j = j0 + e;
          const uint32_t key = key_of(x[e]);
          if (qq < q1 && j >= lo && j < hi && (key & M) == T)
            atomicAdd(hist + ((key >> shift) & nbins_mask), 1u);
        }
      }
    }
  }

  __device__ __forceinline__ int64_t tiles() const { return (q1 - q0 + NT - 1) / NT; }

  __device__ __forceinline__ void tile(int64_t t, uint32_t key[4], int32_t j[4], bool valid[4]) const {
    const int64_t q = q0 + t * NT + threadIdx.x;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q < q1) v = load(q);
    const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int64_t jj = q * 4 - head + e;
      valid[e] = q < q1 && jj >= lo && jj < hi;
      j[e] = (int32_t)jj;
      key[e] = key_of(x[e]);
    }
  }
};

// Per-CTA shared state of the selection.  Everything a peer CTA reads through
// distributed shared memory sits at the same offset in every CTA.
struct SelectShared {
  uint32_t hist1[kBins1];
  uint32_t hist2[kBins23];
  uint32_t hist3[kBins23];
  uint32_t scratch[2][kMaxWarps];
  Pick pick[2];
  uint32_t pub_gt;        // published: this CTA's count of elements above the prefix
  uint32_t pub_eq;        // published: this CTA's count of prefix-equal elements
  uint32_t pub_overflow;  // published: a candidate list overflowed (streaming only)
  uint32_t pub_count;     // published: candidates this CTA listed for the row (streaming only)
};

// Outcome of the selection, identical in every thread of a CTA.
struct Selection {
  uint32_t M, T;   // prefix mask and value of the k-th largest key
  uint32_t quota;  // prefix-equal elements this CTA takes (its first `quota` of them)
  uint32_t off;    // where this CTA's first output goes inside the row
};

// Alternating scratch buffers for the block scans and alternating result
// slots for the bucket picks (two independent counters, so the order in which
// a call's arguments are evaluated does not matter).
struct ScanParity {
  uint32_t p = 0, q = 0;
  __device__ __forceinline__ uint32_t* next(SelectShared& S) {
    uint32_t* s = S.scratch[p];
    p ^= 1u;
    return s;
  }
  __device__ __forceinline__ Pick* next_pick(SelectShared& S) {
    Pick* s = &S.pick[q];
    q ^= 1u;
    return s;
  }
};

// Levels 1..3 of the radix select for one row.  On entry hist1 holds, for
// every bin at or above the row's threshold bin in every CTA of the cluster,
// the exact number of the CTA's elements in that bin, and a barrier (cluster
// barrier with clusters) separates its last update from this call.  `k_row`
// is the number to select (k; the row has more than k elements).
template <int CLUSTER, int NT, class Src>
__device__ __forceinline__ Selection select_levels(SelectShared& S, const Src& src, uint32_t k_row,
                                                   ScanParity& par) {
  Pick pk = block_pick<kBins1, CLUSTER, NT>(S.hist1, k_row, par.next(S), par.next_pick(S));
  uint32_t r = k_row - pk.above;
  uint32_t M = 0xFFF00000u, T = pk.bin << kShift1;
  uint32_t gt = 0, eq = 0;
  if constexpr (CLUSTER > 1) {
    gt = own_above<kBins1, NT>(S.hist1, pk.bin, par.next(S));
    eq = S.hist1[pk.bin];
  }
  if (pk.count != r) {
    // level 2: bits [10, 20) of the keys in bucket T
    for (int b = threadIdx.x; b < kBins23; b += NT) S.hist2[b] = 0u;
    __syncthreads();
    src.histogram(S.hist2, M, T, kShift2, kBins23 - 1);
    __syncthreads();
    if constexpr (CLUSTER > 1) cluster_sync_all();
    pk = block_pick<kBins23, CLUSTER, NT>(S.hist2, r, par.next(S), par.next_pick(S));
    r -= pk.above;
    M |= 0x000FFC00u;
    T |= pk.bin << kShift2;
    if constexpr (CLUSTER > 1) {
      gt += own_above<kBins23, NT>(S.hist2, pk.bin, par.next(S));
      eq = S.hist2[pk.bin];
    }
    if (pk.count != r) {
      // level 3: bits [0, 10)
      for (int b = threadIdx.x; b < kBins23; b += NT) S.hist3[b] = 0u;
      __syncthreads();
      src.histogram(S.hist3, M, T, kShift3, kBins23 - 1);
      __syncthreads();
      if constexpr (CLUSTER > 1) cluster_sync_all();
      pk = block_pick<kBins23, CLUSTER, NT>(S.hist3, r, par.next(S), par.next_pick(S));
      r -= pk.above;
      M = 0xFFFFFFFFu;
      T |= pk.bin;
      if constexpr (CLUSTER > 1) {
        gt += own_above<kBins23, NT>(S.hist3, pk.bin, par.next(S));
        eq = S.hist3[pk.bin];
      }
    }
  }
  Selection sel;
  sel.M = M;
  sel.T = T;
  if constexpr (CLUSTER == 1) {
    sel.quota = r;
    sel.off = 0;
  } else {
    // Tie quota in rank (= window index) order, and each CTA's output offset.
    if (threadIdx.x == 0) {
      S.pub_gt = gt;
      S.pub_eq = eq;
    }
    cluster_sync_all();
    const uint32_t me = cluster_rank();
    uint32_t eq_before = 0, off = 0, quota = 0;
    const uint32_t gt_addr = smem_addr(&S.pub_gt), eq_addr = smem_addr(&S.pub_eq);
    for (uint32_t c = 0; c < (uint32_t)CLUSTER; ++c) {
      const uint32_t gc = ld_cluster_u32(peer_addr(gt_addr, c));
      const uint32_t ec = ld_cluster_u32(peer_addr(eq_addr, c));
      const uint32_t left = r > eq_before ? r - eq_before : 0u;
      const uint32_t qc = ec < left ? ec : left;
      if (c == me) quota = qc;
      if (c < me) off += gc + qc;
      eq_before += ec;
    }
    sel.quota = quota;
    sel.off = off;
  }
  return sel;
}

// Writes, in ascending j, the elements of `src` selected by `sel` to
// out_row[sel.off ...] through the page transform.
template <int NT, class Src>
__device__ __forceinline__ void emit_selected(const Src& src, const Selection& sel, int32_t* out_row,
                                              uint32_t k_row, const int32_t* page_row,
                                              int32_t page_bits, int32_t L, SelectShared& S, ScanParity& par) {
  uint32_t gt_run = 0, eq_run = 0;
  const int64_t nt = src.tiles();
  for (int64_t t = 0; t < nt; ++t) {
    uint32_t key[4];
    int32_t j[4];
    bool valid[4];
    src.tile(t, key, j, valid);
    uint32_t ngt = 0, neq = 0;
    bool is_gt[4], is_eq[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t pk = key[e] & sel.M;
      is_gt[e] = valid[e] && pk > sel.T;
      is_eq[e] = valid[e] && pk == sel.T;
      ngt += is_gt[e];
      neq += is_eq[e];
    }
    uint32_t total;
    const uint32_t ex = block_excl_scan<NT>(ngt | (neq << 16), par.next(S), total);
    uint32_t g = gt_run + (ex & 0xFFFFu), q = eq_run + (ex >> 16);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (is_gt[e] || (is_eq[e] && q < sel.quota)) {
        const uint32_t pos = sel.off + g + (q < sel.quota ? q : sel.quota);
        if (pos < k_row)
          out_row[pos] = page_slot(page_row, page_bits, j[e], L);
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

// A whole row (part) straight from global memory: full level-1 histogram, the
// refinement levels and the emission.  Used by the multipass kernel and by
// the streaming kernel when a row's candidates do not fit its lists.
template <int CLUSTER, int NT>
__device__ __forceinline__ void select_from_global(const Params& p, int32_t row, const Row& r,
                                                   const Part& part, SelectShared& S,
                                                   ScanParity& par) {
  const GlobalSrc<NT> src{r.base4, part.q0, part.q1, r.head, part.lo, part.hi, r.L};
  for (int b = threadIdx.x; b < kBins1; b += NT) S.hist1[b] = 0u;
  __syncthreads();
  src.histogram(S.hist1, 0u, 0u, kShift1, kBins1 - 1);
  __syncthreads();
  if constexpr (CLUSTER > 1) cluster_sync_all();
  const Selection sel = select_levels<CLUSTER, NT>(S, src, (uint32_t)p.k, par);
  emit_selected<NT>(src, sel, p.out + (int64_t)row * p.k, (uint32_t)p.k, r.page_row, p.page_bits, r.L, S, par);
}

}  // namespace topk
