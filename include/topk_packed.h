/*
 * topk_packed.h -- C ABI of the packed-layout top-k + page transform (B300, sm_103a).
 *
 * The operation (page "[sglang] [AMD ROCm] GLM-5.x Prefill 성능을 66% 끌어올린
 * Top-K 커널 최적화 분석", analysis of sglang PR #37889):
 *   - Intro: in the packed DSA prefill layout many requests share one large
 *     score buffer and every row starts at its own column offset;
 *   - section 1 ("TopKPackedParams"): per row i a window length seq_lens[i], a
 *     column offset row_starts[i] and a page-table row row_to_batch[i] (row i
 *     itself when the map is absent); the page-table row starts at
 *     page_table + table_row * stride, and a page transform maps a window index
 *     through it using page_bits;
 *   - section 2 ("Vectorized load alignment and masking"): 16-byte loads start
 *     at a rounded-down address and the lanes before the window are masked so
 *     they never win.  Here the masking is done in registers; the score buffer
 *     is never written.
 * Computed for every row i < num_rows (the page leaves the rule itself
 * unstated; this is the library's specification):
 *     n   = max(seq_lens[i], 0)
 *     v_j = scores[i * row_stride + row_starts[i] + j],   0 <= j < n
 *     S   = the min(k, n) indices j of largest v_j; between equal scores the
 *           lower j is taken (-0.0 and +0.0 are equal)
 *     out[i * k + t] = page_row[j_t >> page_bits] * page_size + (j_t & (page_size - 1))
 *           for the t-th smallest j_t in S, and -1 for min(k, n) <= t < k,
 *     with page_row = page_table + b * pt_stride, b = row_to_batch ? row_to_batch[i] : i,
 *     page_bits = log2(page_size).  Without a page table (page_table NULL) the
 *     transform is the identity: out[i * k + t] = j_t, the raw window index.
 * The result is unique, so it is bit-exact whatever the algorithm.
 */
#ifndef TOPK_PACKED_H_
#define TOPK_PACKED_H_

#include <stdint.h>

#if defined(__GNUC__)
#define TOPK_API __attribute__((visibility("default")))
#else
#define TOPK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream).  NULL is the legacy default stream. */
typedef struct CUstream_st* topk_stream_t;

typedef enum {
  TOPK_OK = 0,
  TOPK_ERR_INVALID_ARG = 1, /* an argument breaks the contract below; nothing launched */
  TOPK_ERR_UNSUPPORTED = 2, /* valid but outside what the library handles (or the chosen kernel
                               cannot be resident on this device); nothing launched */
  TOPK_ERR_LAUNCH = 3,      /* the CUDA launch failed (the CUDA error is kept; see below) */
  TOPK_ERR_DEVICE = 4       /* no usable sm_103a device, or a CUDA query failed */
} topk_status_t;

/* Largest k the library accepts.  Up to TOPK_K_FAST (the sizes the DSA
 * configurations use) the single-pass kernels run; a larger k is served by the
 * multipass kernel, which reads each window several times. */
#define TOPK_K_MAX (1 << 20)
#define TOPK_K_FAST 2048

/*
 * topk_packed -- the operation above, launched asynchronously on `stream`.
 *
 * Arguments (all pointers are DEVICE memory owned by the caller; the library
 * neither frees nor retains them, and allocates nothing):
 *   scores       float32 buffer, read-only, 4-byte aligned; element (i, c) at
 *                scores[i * row_stride + c].
 *   row_stride   elements between consecutive rows of `scores` (>= 0).
 *   seq_lens     int32[num_rows]: window length of each row (negative = 0).
 *   row_starts   int32[num_rows]: window column offset of each row.
 *   row_to_batch int32[num_rows] page-table row of each row, or NULL (identity).
 *   page_table   int32 page numbers; row b starts at page_table + b * pt_stride.  NULL:
 *                no page transform, the output holds raw window indices.
 *   pt_stride    elements between page-table rows (>= 0; 0 lets every row share one).
 *                Not used (nor checked) when page_table is NULL.
 *   page_size    slots per page, a power of two (page_bits = log2(page_size)).  Not
 *                used (nor checked) when page_table is NULL.
 *   k            entries per output row, 1 <= k <= TOPK_K_MAX.
 *   out          int32[num_rows * k], row-major, written completely.
 *   num_rows     number of query rows (>= 0; 0 returns TOPK_OK and launches nothing).
 *   stream       stream to launch on.
 * Preconditions the call cannot check without reading device memory (breaking
 * one gives an unspecified result; reads stay inside the row's window rounded
 * out to 16-byte boundaries, and inside page_row[0 .. ceil(n / page_size))):
 *   0 <= row_starts[i] and row_starts[i] + n <= row_stride for rows read;
 *   page_row covers ceil(n / page_size) pages; page * page_size + page_size - 1 < 2^31;
 *   no NaN inside a window.
 * Returns TOPK_OK once the work is queued.  The call never synchronizes and
 * never reads device arrays on the host.  Errors:
 *   TOPK_ERR_INVALID_ARG  num_rows < 0; k <= 0; row_stride < 0; with a page table,
 *                         page_size <= 0 or not a power of two, or pt_stride < 0;
 *                         scores, seq_lens, row_starts or out NULL while num_rows > 0.
 *   TOPK_ERR_UNSUPPORTED  k > TOPK_K_MAX; scores not 4-byte aligned; with a page
 *                         table, page_size > 2^30; (topk_packed_ex) a k above
 *                         TOPK_K_FAST with the PIPE or SPLIT kernel chosen, or
 *                         the DECODE kernel chosen with row_stride above
 *                         TOPK_DECODE_MAX_STRIDE.
 *   TOPK_ERR_DEVICE       the current device is not sm_103a or cannot be queried.
 *   TOPK_ERR_LAUNCH       the kernel launch was rejected.
 * Thread safety: safe to call from several host threads; calls on different
 * streams may run concurrently.  The only device state they share is the
 * per-device diagnostics word (topk_packed_device_flags), which every launch
 * may set bits in.
 */
TOPK_API topk_status_t topk_packed(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                          const int32_t* row_starts, const int32_t* row_to_batch,
                          const int32_t* page_table, int64_t pt_stride, int32_t page_size,
                          int32_t k, int32_t* out, int32_t num_rows, topk_stream_t stream);

/* Kernel families behind topk_packed_ex. */
typedef enum {
  TOPK_PATH_AUTO = 0,      /* what topk_packed uses (32-bit scores): TOPK_PATH_DECODE when row_stride
                              <= TOPK_DECODE_MAX_STRIDE; TOPK_PATH_STREAM with rows split over a
                              cluster of 2 CTAs (4 when num_rows <= SMs / 4) when row_stride >= 65536
                              and num_rows <= SMs / 2; otherwise, for k <= TOPK_K_FAST,
                              TOPK_PATH_SPLIT (TOPK_PATH_PIPE if the split kernel cannot be resident
                              on the device), and for a larger k TOPK_PATH_MULTIPASS.  16-bit scores:
                              TOPK_PATH_SPLIT */
  TOPK_PATH_MULTIPASS = 1, /* one CTA per row, radix passes straight from global memory */
  TOPK_PATH_STREAM = 2,    /* persistent CTAs, or clusters of 2/4/8 CTAs sharing each row: per-warp
                              TMA rings, a threshold sampled per row that then only rises, per-warp
                              candidate lists; a cluster sums its histograms through distributed
                              shared memory and splits the tie quota by CTA rank */
  TOPK_PATH_PIPE = 3,      /* persistent CTAs, two per SM, 8 warps each: per-warp TMA rings over
                              contiguous blocks of the row, candidates kept in window order with a
                              threshold carried from row to row, ordered emission by prefix counts */
  TOPK_PATH_SPLIT = 4,     /* persistent CTAs, one per SM, each on a contiguous range of rows
                              balanced by cost: 8 streaming warps (8 KB TMA stages, 128 KB in flight
                              per SM) hand each row's candidates, in one of two buffer sets, to 8
                              finishing warps that select and emit it while the next row streams */
  TOPK_PATH_DECODE = 5     /* short windows (row_stride <= TOPK_DECODE_MAX_STRIDE, 32-bit scores):
                              one CTA of 1024 threads per row holds the window in registers and runs
                              an exact radix select on them (a single read of the window) */
} topk_path_t;

/* Largest row_stride TOPK_PATH_DECODE serves. */
#define TOPK_DECODE_MAX_STRIDE 16381

/* Launch choices; zero fields mean "choose automatically". */
typedef struct {
  int32_t path;            /* topk_path_t */
  int32_t cluster_size;    /* STREAM: CTAs that share one row (1, 2, 4 or 8); 0 = auto */
  int32_t max_ctas;        /* STREAM, PIPE, SPLIT, MULTIPASS, DECODE: upper bound on the grid; 0 = auto */
  uint32_t stream_wait_ns; /* PIPE, SPLIT: bound of each wait for a streamed chunk of the window, in
                              ns; 0 = the default of about 2 s.  A wait that runs out sets bit 0 of
                              the diagnostics word; the warp then stops taking chunks and the rows it
                              streams are finished exactly from global memory instead (slower, same
                              result).  The kernel still waits, with the default bound, for every
                              copy it issued before it exits. */
  uint32_t test_flags;     /* 0, or TOPK_TEST_UNSATISFIED_WAIT (for testing the path above): each
                              streaming warp first waits on a barrier that nothing completes, so that
                              the wait runs out after stream_wait_ns.  Other bits: INVALID_ARG. */
  int32_t dependent_launch; /* 1: launch with programmatic stream serialization (programmatic
                              dependent launch), so that the kernel can be scheduled and set up
                              while the previous kernel on `stream` -- typically the one writing the
                              scores -- is still running; it waits for that kernel to complete
                              (griddepcontrol.wait) before reading any argument array, and lets the
                              next kernel on the stream start its own set-up early.  0: an ordinary
                              stream-ordered launch.  Other values: INVALID_ARG.  (Page section 2,
                              PDLWaitPrimary before the scores are read.) */
} topk_launch_config_t;

#define TOPK_TEST_UNSATISFIED_WAIT 1u

/*
 * topk_packed_ex -- topk_packed with explicit launch choices.  `config` may be
 * NULL (same as topk_packed).  Every path computes the same, bit-identical
 * result.  Extra error: TOPK_ERR_INVALID_ARG for an unknown path or a
 * cluster_size other than 0, 1, 2, 4, 8.
 */
TOPK_API topk_status_t topk_packed_ex(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                             const int32_t* row_starts, const int32_t* row_to_batch,
                             const int32_t* page_table, int64_t pt_stride, int32_t page_size,
                             int32_t k, int32_t* out, int32_t num_rows,
                             const topk_launch_config_t* config, topk_stream_t stream);

/* Element types of a score buffer (topk_packed_typed). */
typedef enum {
  TOPK_F32 = 0,  /* IEEE binary32 (float), as in topk_packed */
  TOPK_BF16 = 1, /* bfloat16: the upper 16 bits of a binary32 */
  TOPK_F16 = 2   /* IEEE binary16 (half) */
} topk_dtype_t;

/*
 * topk_packed_typed -- topk_packed_ex on a score buffer of `dtype` elements
 * (topk_dtype_t): element (i, c) at ((const T*)scores)[i * row_stride + c],
 * row_stride and row_starts counted in elements.  A 16-bit buffer halves the
 * bytes read; the selection is that of the same values held as 32-bit floats
 * (every bfloat16 and binary16 value is exactly a binary32 value; -0.0 and
 * +0.0 are equal; NaN outside the contract).  The page's TopKPackedParams
 * (section 1) declares the buffer as float*; the 16-bit types are this
 * library's extension.
 * Extra errors: TOPK_ERR_INVALID_ARG for an unknown dtype; TOPK_ERR_UNSUPPORTED
 * for scores not aligned to the element size, and, for a 16-bit dtype, a k
 * above TOPK_K_FAST or a kernel family other than AUTO and SPLIT.
 */
TOPK_API topk_status_t topk_packed_typed(const void* scores, int32_t dtype, int64_t row_stride,
                                         const int32_t* seq_lens, const int32_t* row_starts,
                                         const int32_t* row_to_batch, const int32_t* page_table,
                                         int64_t pt_stride, int32_t page_size, int32_t k, int32_t* out,
                                         int32_t num_rows, const topk_launch_config_t* config,
                                         topk_stream_t stream);

/*
 * topk_packed_plan -- the launch topk_packed_ex would make for these sizes,
 * without launching: path, cluster size, grid (in CTAs) and threads per CTA.
 * Any output pointer may be NULL.  Errors as topk_packed_ex (no pointer checks).
 */
TOPK_API topk_status_t topk_packed_plan(int64_t row_stride, int32_t k, int32_t num_rows,
                               const topk_launch_config_t* config, int32_t* path,
                               int32_t* cluster_size, int32_t* grid_ctas,
                               int32_t* threads_per_cta);

/* Static description of a status code (never NULL). */
TOPK_API const char* topk_status_string(topk_status_t status);

/* The CUDA error code (cudaError_t as int) behind the last TOPK_ERR_LAUNCH or
 * TOPK_ERR_DEVICE returned on the calling host thread, 0 if none. */
TOPK_API int topk_last_cuda_error(void);

/*
 * Device-side diagnostics: one 32-bit word per device, shared by every launch
 * of the library on that device (whatever the stream).  Every wait inside the
 * kernels is bounded; a wait that runs out records a bit here instead of
 * hanging, and the kernel finishes its control flow:
 *   bit 0: a wait for a TMA chunk of the score stream gave up.  In the PIPE and
 *          SPLIT kernels the affected rows are then finished exactly from
 *          global memory (same result, slower); in the others they are
 *          unspecified.  Every copy a kernel issued has landed before it exits.
 *   bit 1: an output position at or past k was computed (a selection that is
 *          not exact); the position is not written.  Never expected.
 *   bit 2 and bits 8-15 (only in libtopk_packed_checked.so, the same library
 *          compiled with TOPK_CHECKED for testing): a bounds check failed.
 *          That build checks, at run time, every global-memory address it
 *          computes (window loads and bulk copies against the row's window
 *          rounded out to 16 bytes, page-table reads against the window
 *          length, descriptor reads against num_rows) and every shared-memory
 *          index that is not in range by construction; a failed check sets
 *          bit 2, the access is skipped, and bits 8-15 keep the site of the
 *          first failure:
 *            1 a row's window leaves its buffer row (the precondition
 *              row_starts[i] + n <= row_stride; recorded, the row still read),
 *            2 a descriptor read for a row outside [0, num_rows),
 *            3 a window load, 4 a window bulk copy, 5 a page-table read
 *              outside the window, 6 a shared page-stage read, 7 a candidate
 *              store, 8 a region or list count, 9 a staged output position,
 *              10 a sample load.
 *          The normal library compiles every check away.
 * topk_packed_device_flags copies the word of the current device into *flags
 * (after the work queued on `stream` so far) and, when `reset` is non-zero,
 * clears it.  It synchronizes `stream`.  A reset races with launches running
 * on other streams of the same device: a bit one of them sets between the
 * copy and the clear is lost, so read with reset only when no other launch
 * is in flight.
 */
TOPK_API topk_status_t topk_packed_device_flags(uint32_t* flags, int32_t reset, topk_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TOPK_PACKED_H_ */
