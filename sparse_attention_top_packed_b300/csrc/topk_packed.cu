// C ABI of the packed top-k + page transform: argument checks, launch planning
// and kernel launches.  Declarations and the contract: include/topk_packed.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "topk_decode.cuh"
#include "topk_kernels.cuh"
#include "topk_pipe.cuh"
#include "topk_split.cuh"
#include "topk_packed.h"

namespace {

using topk::Params;

thread_local int g_last_cuda_error = 0;

topk_status_t cuda_fail(cudaError_t e, topk_status_t s) {
  g_last_cuda_error = (int)e;
  return s;
}

constexpr int kMaxDevices = 64;

// Per-device facts and one-time kernel attributes.
struct DeviceInfo {
  bool ok = false;
  int sms = 0;
  int stream_ctas_per_sm = 0;     // resident stream CTAs per SM (cluster size 1)
  int stream_clusters[4] = {};    // max resident clusters for sizes 2, 4, 8 (index 1..3)
  int multipass_ctas_per_sm = 0;
  int pipe_ctas_per_sm = 0;
  int split_ctas_per_sm = 0;
  int decode_ctas_per_sm = 0;
  cudaError_t error = cudaSuccess;
};

std::once_flag g_once[kMaxDevices];
DeviceInfo g_info[kMaxDevices];

template <int C>
cudaError_t prepare_stream(int& occupancy_or_clusters, int sms) {
  const size_t smem = sizeof(topk::StreamShared);
  cudaError_t e = cudaFuncSetAttribute(topk::topk_stream_kernel<C>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if constexpr (C == 1) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occupancy_or_clusters,
                                                         topk::topk_stream_kernel<1>, topk::kStreamThreads, smem);
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(C * sms), 1, 1);
    cfg.blockDim = dim3(topk::kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(&occupancy_or_clusters, topk::topk_stream_kernel<C>, &cfg);
  }
}

void init_device(int dev) {
  DeviceInfo& d = g_info[dev];
  cudaDeviceProp prop;
  cudaError_t e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) {
    d.error = e;
    return;
  }
  if (prop.major != 10 || prop.minor != 3) {
    d.error = cudaErrorNoKernelImageForDevice;
    return;
  }
  d.sms = prop.multiProcessorCount;
  const size_t mp_smem = sizeof(topk::SelectShared);
  e = cudaFuncSetAttribute(topk::topk_multipass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)mp_smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.multipass_ctas_per_sm, topk::topk_multipass_kernel,
                                                      topk::kMultipassThreads, mp_smem);
  const size_t pipe_smem = sizeof(topk::pipe::PipeSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(topk::pipe::topk_pipe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pipe_smem);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.pipe_ctas_per_sm, topk::pipe::topk_pipe_kernel,
                                                      topk::pipe::kBlock, pipe_smem);
  if (e == cudaSuccess) {
    // the split kernel is optional: if it cannot be made resident, its path
    // reports TOPK_ERR_UNSUPPORTED and the others are unaffected
    using topk::ElemBF16;
    using topk::ElemF16;
    using topk::ElemF32;
    using topk::split::SplitSmem;
    cudaError_t es = cudaFuncSetAttribute(topk::split::topk_split_kernel<ElemF32>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(SplitSmem<ElemF32>));
    if (es == cudaSuccess)
      es = cudaFuncSetAttribute(topk::split::topk_split_kernel<ElemBF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(SplitSmem<ElemBF16>));
    if (es == cudaSuccess)
      es = cudaFuncSetAttribute(topk::split::topk_split_kernel<ElemF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sizeof(SplitSmem<ElemF16>));
    if (es == cudaSuccess)
      es = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.split_ctas_per_sm, topk::split::topk_split_kernel<ElemBF16>,
                                                         topk::split::kBlockThreads, sizeof(SplitSmem<ElemBF16>));
    if (es != cudaSuccess) {
      d.split_ctas_per_sm = 0;
      (void)cudaGetLastError();  // clear it: the other kernels stay usable
    }
  }
  if (e == cudaSuccess) {
    const int ss = (int)sizeof(topk::SelectShared);
    e = cudaFuncSetAttribute(topk::decode::topk_decode_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, ss);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(topk::decode::topk_decode_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, ss);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(topk::decode::topk_decode_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, ss);
    if (e == cudaSuccess)
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&d.decode_ctas_per_sm, topk::decode::topk_decode_kernel<4>,
                                                        topk::decode::kThreads, ss);
  }
  if (e == cudaSuccess) e = prepare_stream<1>(d.stream_ctas_per_sm, d.sms);
  if (e == cudaSuccess) e = prepare_stream<2>(d.stream_clusters[1], d.sms);
  if (e == cudaSuccess) e = prepare_stream<4>(d.stream_clusters[2], d.sms);
  if (e == cudaSuccess) e = prepare_stream<8>(d.stream_clusters[3], d.sms);
  if (e != cudaSuccess) {
    d.error = e;
    return;
  }
  d.ok = d.multipass_ctas_per_sm > 0 && d.stream_ctas_per_sm > 0 && d.pipe_ctas_per_sm > 0 &&
         d.decode_ctas_per_sm > 0;
  if (!d.ok) d.error = cudaErrorInvalidConfiguration;
}

const DeviceInfo* device_info(topk_status_t& st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    st = cuda_fail(e == cudaSuccess ? cudaErrorInvalidDevice : e, TOPK_ERR_DEVICE);
    return nullptr;
  }
  std::call_once(g_once[dev], init_device, dev);
  if (!g_info[dev].ok) {
    st = cuda_fail(g_info[dev].error, TOPK_ERR_DEVICE);
    return nullptr;
  }
  return &g_info[dev];
}

struct Plan {
  int32_t path;
  int32_t cluster;
  int64_t grid;
};

int log2_exact(int32_t v) {
  int b = 0;
  while ((1 << b) < v) ++b;
  return b;
}

// `has_table`: a page table is given (without one, page_size and pt_stride
// are not used and not checked).
topk_status_t check_sizes(int64_t row_stride, int64_t pt_stride, int32_t page_size, int32_t k,
                          int32_t num_rows, const topk_launch_config_t* cfg, bool has_table) {
  if (num_rows < 0 || k <= 0 || row_stride < 0) return TOPK_ERR_INVALID_ARG;
  if (has_table && (pt_stride < 0 || page_size <= 0 || (page_size & (page_size - 1)) != 0))
    return TOPK_ERR_INVALID_ARG;
  if (cfg) {
    if (cfg->path < TOPK_PATH_AUTO || cfg->path > TOPK_PATH_DECODE) return TOPK_ERR_INVALID_ARG;
    const int c = cfg->cluster_size;
    if (!(c == 0 || c == 1 || c == 2 || c == 4 || c == 8)) return TOPK_ERR_INVALID_ARG;
    if (cfg->max_ctas < 0) return TOPK_ERR_INVALID_ARG;
    if ((cfg->test_flags & ~(uint32_t)TOPK_TEST_UNSATISFIED_WAIT) != 0u) return TOPK_ERR_INVALID_ARG;
    if (cfg->dependent_launch != 0 && cfg->dependent_launch != 1) return TOPK_ERR_INVALID_ARG;
  }
  if (k > TOPK_K_MAX) return TOPK_ERR_UNSUPPORTED;
  if (has_table && page_size > (1 << 30)) return TOPK_ERR_UNSUPPORTED;
  return TOPK_OK;
}

int cluster_index(int c) { return c == 2 ? 1 : c == 4 ? 2 : 3; }

// Shortest row_stride for which the automatic choice splits rows over a cluster.
constexpr int64_t kClusterMinStride = 65536;

static_assert(topk::decode::max_stride<4>() == TOPK_DECODE_MAX_STRIDE, "decode kernel bound");

// Quads a thread of the decode kernel holds for this row_stride (1, 2 or 4).
int decode_qpt(int64_t row_stride) {
  return row_stride <= topk::decode::max_stride<1>() ? 1 : row_stride <= topk::decode::max_stride<2>() ? 2 : 4;
}

Plan make_plan(const DeviceInfo& d, int64_t row_stride, int32_t k, int32_t num_rows,
               const topk_launch_config_t* cfg, bool f32) {
  Plan pl;
  const int32_t want = cfg ? cfg->path : TOPK_PATH_AUTO;
  // short windows: the register-resident decode kernel (a row's time is
  // latency there); otherwise the warp-specialised split kernel, whose stream
  // never waits for the end of a row; the pipelined kernel when the split one
  // cannot be resident; the multipass kernel for a k beyond the single-pass
  // kernels' buffers
  // long windows in a batch of at most half as many rows as SMs: each row
  // split over a cluster (2 CTAs, or 4 up to a quarter as many rows as SMs)
  // that merges its histograms through distributed shared memory
  int auto_cluster = 0;
  if (want != TOPK_PATH_AUTO)
    pl.path = want;
  else if (f32 && row_stride <= TOPK_DECODE_MAX_STRIDE)
    pl.path = TOPK_PATH_DECODE;
  else if (f32 && row_stride >= kClusterMinStride && 2 * (int64_t)num_rows <= d.sms &&
           d.stream_clusters[cluster_index(2)] > 0) {
    pl.path = TOPK_PATH_STREAM;
    auto_cluster = 4 * (int64_t)num_rows <= d.sms && d.stream_clusters[cluster_index(4)] > 0 ? 4 : 2;
  } else if (k > TOPK_K_FAST)
    pl.path = TOPK_PATH_MULTIPASS;
  else
    pl.path = d.split_ctas_per_sm > 0 ? TOPK_PATH_SPLIT : TOPK_PATH_PIPE;
  pl.cluster = 1;
  if (pl.path == TOPK_PATH_DECODE) {
    const int64_t cap = (int64_t)d.sms * d.decode_ctas_per_sm;
    pl.grid = num_rows < cap ? num_rows : cap;
    if (cfg && cfg->max_ctas > 0 && pl.grid > cfg->max_ctas) pl.grid = cfg->max_ctas;
    return pl;
  }
  if (pl.path == TOPK_PATH_PIPE) {
    const int64_t cap = (int64_t)d.sms * d.pipe_ctas_per_sm;
    pl.grid = num_rows < cap ? num_rows : cap;
    if (cfg && cfg->max_ctas > 0 && pl.grid > cfg->max_ctas) pl.grid = cfg->max_ctas;
    return pl;
  }
  if (pl.path == TOPK_PATH_SPLIT) {
    const int64_t cap = (int64_t)d.sms * d.split_ctas_per_sm;
    pl.grid = num_rows < cap ? num_rows : cap;
    if (cfg && cfg->max_ctas > 0 && pl.grid > cfg->max_ctas) pl.grid = cfg->max_ctas;
    return pl;
  }
  if (pl.path == TOPK_PATH_MULTIPASS) {
    const int64_t cap = (int64_t)d.sms * d.multipass_ctas_per_sm * 8;
    pl.grid = num_rows < cap ? num_rows : cap;
    if (cfg && cfg->max_ctas > 0 && pl.grid > cfg->max_ctas) pl.grid = cfg->max_ctas;
    return pl;
  }
  pl.cluster = (cfg && cfg->cluster_size > 0) ? cfg->cluster_size : auto_cluster > 0 ? auto_cluster : 1;
  int64_t clusters;
  if (pl.cluster == 1) {
    clusters = (int64_t)d.sms * d.stream_ctas_per_sm;
  } else {
    clusters = d.stream_clusters[cluster_index(pl.cluster)];
    if (clusters <= 0) clusters = 1;
  }
  if (clusters > num_rows) clusters = num_rows;
  if (cfg && cfg->max_ctas > 0) {
    const int64_t lim = cfg->max_ctas / pl.cluster;
    if (clusters > lim) clusters = lim > 0 ? lim : 1;
  }
  pl.grid = clusters * pl.cluster;
  return pl;
}

// One launch through cudaLaunchKernelEx: optional thread-block cluster and
// programmatic stream serialization (the kernel may start while the previous
// kernel on the stream still runs; it waits for it before reading inputs).
template <class Kernel>
cudaError_t launch(Kernel kernel, int64_t grid, int threads, size_t smem, int cluster, bool dependent,
                   cudaStream_t stream, const Params& prm) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3((unsigned)threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (dependent) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = n ? attr : nullptr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, prm);
}

static_assert(topk::pipe::kKMax == TOPK_K_FAST, "the single-pass kernels are sized for TOPK_K_FAST");

}  // namespace

extern "C" {

topk_status_t topk_packed_typed(const void* scores, int32_t dtype, int64_t row_stride, const int32_t* seq_lens,
                                const int32_t* row_starts, const int32_t* row_to_batch,
                                const int32_t* page_table, int64_t pt_stride, int32_t page_size,
                                int32_t k, int32_t* out, int32_t num_rows,
                                const topk_launch_config_t* config, topk_stream_t stream) {
  g_last_cuda_error = 0;
  if (dtype != TOPK_F32 && dtype != TOPK_BF16 && dtype != TOPK_F16) return TOPK_ERR_INVALID_ARG;
  topk_status_t st = check_sizes(row_stride, pt_stride, page_size, k, num_rows, config, page_table != nullptr);
  if (st != TOPK_OK) return st;
  const bool half = dtype != TOPK_F32;
  const int32_t want = config ? config->path : TOPK_PATH_AUTO;
  if (half && ((want != TOPK_PATH_AUTO && want != TOPK_PATH_SPLIT) || k > TOPK_K_FAST)) return TOPK_ERR_UNSUPPORTED;
  if (num_rows == 0) return TOPK_OK;
  if (!scores || !seq_lens || !row_starts || !out) return TOPK_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(scores) & (half ? 1u : 3u)) != 0) return TOPK_ERR_UNSUPPORTED;
  const DeviceInfo* d = device_info(st);
  if (!d) return st;

  Params prm;
  prm.scores = static_cast<const float*>(scores);  // element type: dtype
  prm.row_stride = row_stride;
  prm.seq_lens = seq_lens;
  prm.row_starts = row_starts;
  prm.row_to_batch = row_to_batch;
  prm.page_table = page_table;
  prm.pt_stride = page_table ? pt_stride : 0;
  prm.page_bits = page_table ? log2_exact(page_size) : 0;
  prm.k = k;
  prm.out = out;
  prm.num_rows = num_rows;
  prm.stream_wait_ns = config ? config->stream_wait_ns : 0u;
  prm.test_flags = config ? config->test_flags : 0u;

  const Plan pl = make_plan(*d, row_stride, k, num_rows, config, !half);
  if (pl.grid <= 0) return TOPK_ERR_UNSUPPORTED;  // the split kernel cannot be resident here
  if (k > TOPK_K_FAST && (pl.path == TOPK_PATH_PIPE || pl.path == TOPK_PATH_SPLIT)) return TOPK_ERR_UNSUPPORTED;
  if (pl.path == TOPK_PATH_DECODE && row_stride > TOPK_DECODE_MAX_STRIDE) return TOPK_ERR_UNSUPPORTED;
  if (half && pl.path != TOPK_PATH_SPLIT) return TOPK_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool dep = config && config->dependent_launch != 0;
  cudaError_t e;
  if (pl.path == TOPK_PATH_PIPE) {
    e = launch(topk::pipe::topk_pipe_kernel, pl.grid, topk::pipe::kBlock, sizeof(topk::pipe::PipeSmem), 1, dep, s,
               prm);
  } else if (pl.path == TOPK_PATH_SPLIT) {
    using topk::split::SplitSmem;
    using topk::split::topk_split_kernel;
    const int nt = topk::split::kBlockThreads;
    if (dtype == TOPK_BF16)
      e = launch(topk_split_kernel<topk::ElemBF16>, pl.grid, nt, sizeof(SplitSmem<topk::ElemBF16>), 1, dep, s, prm);
    else if (dtype == TOPK_F16)
      e = launch(topk_split_kernel<topk::ElemF16>, pl.grid, nt, sizeof(SplitSmem<topk::ElemF16>), 1, dep, s, prm);
    else
      e = launch(topk_split_kernel<topk::ElemF32>, pl.grid, nt, sizeof(SplitSmem<topk::ElemF32>), 1, dep, s, prm);
  } else if (pl.path == TOPK_PATH_MULTIPASS) {
    e = launch(topk::topk_multipass_kernel, pl.grid, topk::kMultipassThreads, sizeof(topk::SelectShared), 1, dep, s,
               prm);
  } else if (pl.path == TOPK_PATH_DECODE) {
    const size_t ss = sizeof(topk::SelectShared);
    const int nt = topk::decode::kThreads, qpt = decode_qpt(row_stride);
    if (qpt == 1)
      e = launch(topk::decode::topk_decode_kernel<1>, pl.grid, nt, ss, 1, dep, s, prm);
    else if (qpt == 2)
      e = launch(topk::decode::topk_decode_kernel<2>, pl.grid, nt, ss, 1, dep, s, prm);
    else
      e = launch(topk::decode::topk_decode_kernel<4>, pl.grid, nt, ss, 1, dep, s, prm);
  } else {
    const size_t sm = sizeof(topk::StreamShared);
    switch (pl.cluster) {
      case 1: e = launch(topk::topk_stream_kernel<1>, pl.grid, topk::kStreamThreads, sm, 1, dep, s, prm); break;
      case 2: e = launch(topk::topk_stream_kernel<2>, pl.grid, topk::kStreamThreads, sm, 2, dep, s, prm); break;
      case 4: e = launch(topk::topk_stream_kernel<4>, pl.grid, topk::kStreamThreads, sm, 4, dep, s, prm); break;
      default: e = launch(topk::topk_stream_kernel<8>, pl.grid, topk::kStreamThreads, sm, 8, dep, s, prm); break;
    }
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, TOPK_ERR_LAUNCH);
  return TOPK_OK;
}

topk_status_t topk_packed_ex(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                             const int32_t* row_starts, const int32_t* row_to_batch,
                             const int32_t* page_table, int64_t pt_stride, int32_t page_size,
                             int32_t k, int32_t* out, int32_t num_rows,
                             const topk_launch_config_t* config, topk_stream_t stream) {
  return topk_packed_typed(scores, TOPK_F32, row_stride, seq_lens, row_starts, row_to_batch, page_table, pt_stride,
                           page_size, k, out, num_rows, config, stream);
}

topk_status_t topk_packed(const float* scores, int64_t row_stride, const int32_t* seq_lens,
                          const int32_t* row_starts, const int32_t* row_to_batch,
                          const int32_t* page_table, int64_t pt_stride, int32_t page_size,
                          int32_t k, int32_t* out, int32_t num_rows, topk_stream_t stream) {
  return topk_packed_ex(scores, row_stride, seq_lens, row_starts, row_to_batch, page_table, pt_stride,
                        page_size, k, out, num_rows, nullptr, stream);
}

topk_status_t topk_packed_plan(int64_t row_stride, int32_t k, int32_t num_rows,
                               const topk_launch_config_t* config, int32_t* path,
                               int32_t* cluster_size, int32_t* grid_ctas, int32_t* threads_per_cta) {
  g_last_cuda_error = 0;
  topk_status_t st = check_sizes(row_stride, 0, 1, k, num_rows, config, true);
  if (st != TOPK_OK) return st;
  const DeviceInfo* d = device_info(st);
  if (!d) return st;
  const Plan pl = make_plan(*d, row_stride, k, num_rows, config, true);
  if (pl.grid <= 0 && num_rows > 0) return TOPK_ERR_UNSUPPORTED;
  if (k > TOPK_K_FAST && (pl.path == TOPK_PATH_PIPE || pl.path == TOPK_PATH_SPLIT)) return TOPK_ERR_UNSUPPORTED;
  if (pl.path == TOPK_PATH_DECODE && row_stride > TOPK_DECODE_MAX_STRIDE) return TOPK_ERR_UNSUPPORTED;
  if (path) *path = pl.path;
  if (cluster_size) *cluster_size = pl.cluster;
  if (grid_ctas) *grid_ctas = (int32_t)pl.grid;
  if (threads_per_cta)
    *threads_per_cta = pl.path == TOPK_PATH_PIPE        ? topk::pipe::kBlock
                       : pl.path == TOPK_PATH_SPLIT     ? topk::split::kBlockThreads
                       : pl.path == TOPK_PATH_MULTIPASS ? topk::kMultipassThreads
                       : pl.path == TOPK_PATH_DECODE    ? topk::decode::kThreads
                                                        : topk::kStreamThreads;
  return TOPK_OK;
}

const char* topk_status_string(topk_status_t status) {
  switch (status) {
    case TOPK_OK: return "success";
    case TOPK_ERR_INVALID_ARG: return "invalid argument";
    case TOPK_ERR_UNSUPPORTED: return "unsupported argument for this library";
    case TOPK_ERR_LAUNCH: return "kernel launch failed";
    case TOPK_ERR_DEVICE: return "no usable sm_103a device";
  }
  return "unknown status";
}

int topk_last_cuda_error(void) { return g_last_cuda_error; }

topk_status_t topk_packed_device_flags(uint32_t* flags, int32_t reset, topk_stream_t stream) {
  g_last_cuda_error = 0;
  if (!flags) return TOPK_ERR_INVALID_ARG;
  topk_status_t st;
  if (!device_info(st)) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyFromSymbolAsync(flags, topk::g_device_flags, sizeof(uint32_t), 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess && reset) {
    static const uint32_t zero = 0;
    e = cudaMemcpyToSymbolAsync(topk::g_device_flags, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, s);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, TOPK_ERR_DEVICE);
  return TOPK_OK;
}

}  // extern "C"
