// api.cu -- the C ABI declared in include/softmax_rows.h.
//
// Host side only: argument validation, per-device properties, variant choice, the per-device
// status word, and the host-buffer pipeline.  Every step of the computation runs in the
// kernels of kernels_rowwise.cu, kernel_oneread_tma.cu and kernel_splitrow.cu.
#include <cmath>
#include <mutex>
#include <string>

#include "../../include/softmax_rows.h"
#include "attention.h"
#include "launch.h"

namespace rwo {

__device__ unsigned g_status;  // per-device status word (kernels atomicOr status bits into it)

namespace {

bool cluster_local_rows(const RowProblem& p, const DeviceInfo& dev);

constexpr int kMaxDevices = 64;

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices];

thread_local std::string t_last_cuda_error;
thread_local int t_last_variant = SOFTMAX_VARIANT_AUTO;

uint64_t g_exchange_wait_ns = 200ull * 1000 * 1000;  // 200 ms
int g_debug_fault = 0;
std::mutex g_debug_mutex;

// Per-device resources of softmax_rows_host, created on first use and kept for the life of the
// process: copy/compute lanes (non-blocking streams), events and grow-only staging buffers.
struct HostPipe {
  static constexpr int kLanes = 3;
  std::mutex mu;
  bool ready = false;
  cudaStream_t lanes[kLanes] = {};
  cudaEvent_t ev_start = nullptr;
  cudaEvent_t ev_done[kLanes] = {};
  void* buf[kLanes] = {};
  size_t buf_bytes = 0;

  cudaError_t prepare(size_t bytes) {
    cudaError_t err;
    if (!ready) {
      for (int i = 0; i < kLanes; ++i) {
        if ((err = cudaStreamCreateWithFlags(&lanes[i], cudaStreamNonBlocking)) != cudaSuccess) return err;
        if ((err = cudaEventCreateWithFlags(&ev_done[i], cudaEventDisableTiming)) != cudaSuccess) return err;
      }
      if ((err = cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming)) != cudaSuccess) return err;
      ready = true;
    }
    if (bytes > buf_bytes) {
      for (int i = 0; i < kLanes; ++i) {
        if (buf[i]) {
          if ((err = cudaStreamSynchronize(lanes[i])) != cudaSuccess) return err;
          if ((err = cudaFree(buf[i])) != cudaSuccess) return err;
          buf[i] = nullptr;
        }
      }
      buf_bytes = 0;
      for (int i = 0; i < kLanes; ++i)
        if ((err = cudaMalloc(&buf[i], bytes)) != cudaSuccess) return err;
      buf_bytes = bytes;
    }
    return cudaSuccess;
  }
};
HostPipe g_pipe[kMaxDevices];

int cuda_fail(cudaError_t err) {
  t_last_cuda_error = cudaGetErrorString(err);
  return SOFTMAX_ERR_CUDA;
}

// Properties of the current device, queried once per device.
int current_device_info(const DeviceInfo** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err);
  if (dev < 0 || dev >= kMaxDevices) return cuda_fail(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (!g_dev_ready[dev]) {
    DeviceInfo info;
    info.device = dev;
    if ((err = cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&info.max_smem_per_block_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                      dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&info.max_smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess ||
        (err = cudaDeviceGetAttribute(&info.max_threads_per_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) !=
            cudaSuccess ||
        (err = cudaDeviceGetAttribute(&info.l2_bytes, cudaDevAttrL2CacheSize, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&info.cluster_launch, cudaDevAttrClusterLaunch, dev)) != cudaSuccess)
      return cuda_fail(err);
    void* status = nullptr;
    if ((err = cudaGetSymbolAddress(&status, g_status)) != cudaSuccess) return cuda_fail(err);
    info.status = static_cast<unsigned*>(status);
    g_dev[dev] = info;
    g_dev_ready[dev] = true;
  }
  *out = &g_dev[dev];
  return SOFTMAX_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape and pointer checks shared by the row calls.  Returns a status; sets *noop for M == 0.
int validate_rows(const void* x, int64_t M, int64_t N, int dtype, bool* noop) {
  *noop = false;
  if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_BF16 && dtype != SOFTMAX_F16) return SOFTMAX_ERR_INVALID_ARG;
  if (N < 1 || M < 0) return SOFTMAX_ERR_INVALID_ARG;
  const int64_t s = elem_bytes(dtype);
  if (N > INT64_MAX / s) return SOFTMAX_ERR_INVALID_ARG;
  if (M == 0) {  // nothing to do; pointers of an empty matrix may be NULL
    *noop = true;
    return SOFTMAX_OK;
  }
  if (M > INT64_MAX / (N * s)) return SOFTMAX_ERR_INVALID_ARG;
  if (!x) return SOFTMAX_ERR_INVALID_ARG;
  return SOFTMAX_OK;
}

// Aligned rows above this length take the cluster-row kernel for the two passes (clusters of one
// CTA up to ~260 KiB rows, larger ones beyond, so that the rows in flight stay within L2); the
// two-pass kernel keeps shorter and unaligned rows, whose thread count it sizes to the row.
constexpr int64_t kClusterRowMinBytes = int64_t(64) << 10;

cudaError_t launch_twopass_any(const RowProblem& p, bool aligned, const DeviceInfo& dev) {
  if (aligned && p.N * elem_bytes(p.dtype) > kClusterRowMinBytes && clusterrow_fits(p, dev))
    return launch_clusterrow(p, dev);
  return launch_twopass(p, aligned, dev);
}

int run_variant(RowProblem& p, int variant, const DeviceInfo& dev) {
  const bool aligned = aligned16(p.x) && (p.y == nullptr || aligned16(p.y)) &&
                       (p.N * elem_bytes(p.dtype)) % 16 == 0;
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  if (variant == SOFTMAX_VARIANT_AUTO) {
    if (aligned) {
      // Measured on GB300 (~1 GB per launch): the register kernel for every fp32 row up to 64 KiB
      // (4-8 KiB 6.95 TB/s against 5.78-6.21 on the warp-per-row bulk-copy kernel, 20-32 KiB
      // 6.87-6.90 against 5.69-5.92 on the CTA bulk-copy kernel, 40 KiB 6.88 against 6.54, 48 KiB
      // 6.88 against 5.96, 56 KiB 6.86 against 5.79 on two passes, 64 KiB 6.88 against 6.21) and
      // for 16-bit rows up to 4 KiB (bf16 4 KiB 6.22 against 5.95); the warp-per-row kernel for
      // many 16-bit rows of 4-8 KiB (bf16 8 KiB 6.52 against 5.84 in registers); the CTA
      // bulk-copy kernel for longer 16-bit rows (registers there: bf16 12 / 16 KiB 5.32 / 5.48
      // against 6.50 / 6.63 with x kept packed, 24-32 KiB 4.8-4.9 against 5.9-6.0, 48 KiB 5.08
      // against 6.89, 64 KiB 3.94 against 6.70).
      const bool f32 = p.dtype == SOFTMAX_F32;
      if (!f32 && row_bytes > 4096 && row_bytes <= 8192 && p.M >= 4 * int64_t(dev.sm_count) &&
          oneread_warp_fits(p, dev))
        variant = SOFTMAX_VARIANT_ONEREAD_SMEM;
      else if (row_bytes <= (f32 ? 65536 : 8192) && oneread_reg_fits(p, true))
        variant = SOFTMAX_VARIANT_ONEREAD_REG;
      else if (oneread_tma_fits(p, dev))
        variant = SOFTMAX_VARIANT_ONEREAD_SMEM;
      else if (!p.shares_gpu && (row_bytes >= (int64_t(8) << 20) || (row_bytes >= (int64_t(4) << 20) && p.M <= 16)) &&
               splitrow_fits(p, dev))
        // rows of 8 MiB and more at any count, and rows of 4 MiB and more when there are at most
        // 16: one row over the whole GPU, each CTA's segment held on chip where it fits (measured,
        // fp32, split row against the cluster-row two passes: 32 x 16 MiB 163 against 272 us,
        // 300 x 8 MiB 869 against 1076, 16 x 4 MiB 36.6 against 41.2; but 64 x 4 MiB 133 against
        // 116, 8 x 2 MiB 20.8 against 17.1, 76 x 1 MiB 124 against 44.5: there each row's
        // exchange costs more than the clusters' parallel rows)
        variant = SOFTMAX_VARIANT_SPLITROW;
      else if (cluster_local_rows(p, dev))
        variant = SOFTMAX_VARIANT_ONEREAD_SMEM;
      else
        variant = SOFTMAX_VARIANT_TWOPASS;
    } else {
      variant = (p.N <= 512 && oneread_reg_fits(p, false)) ? SOFTMAX_VARIANT_ONEREAD_REG
                                                           : SOFTMAX_VARIANT_TWOPASS;
    }
  }
  cudaError_t err;
  switch (variant) {
    case SOFTMAX_VARIANT_ONEREAD_REG:
      if (!oneread_reg_fits(p, aligned)) return SOFTMAX_ERR_UNSUPPORTED;
      err = launch_oneread_reg(p, aligned, dev);
      break;
    case SOFTMAX_VARIANT_ONEREAD_SMEM:
      if (!aligned) return SOFTMAX_ERR_MISALIGNED;
      // rows up to 8 KiB: one warp per row; longer rows: the CTA bulk-copy kernel (measured on
      // 4096 x 4096 fp32: 23.7 us against 25.3 us for the warp kernel); the warp kernel again
      // where the bulk-copy kernel does not fit
      if (p.N * elem_bytes(p.dtype) <= 8192 && oneread_warp_fits(p, dev))
        err = launch_oneread_warp(p, dev);
      else if (oneread_tma_fits(p, dev))
        err = launch_oneread_tma(p, dev);
      else if (oneread_warp_fits(p, dev))
        err = launch_oneread_warp(p, dev);
      else if (clusterrow_onchip_fits(p, dev))  // rows above 64 KiB: a cluster per row, held on chip
        err = launch_clusterrow_onchip(p, dev);
      else
        return SOFTMAX_ERR_UNSUPPORTED;
      break;
    case SOFTMAX_VARIANT_TWOPASS:
      err = launch_twopass_any(p, aligned, dev);
      break;
    case SOFTMAX_VARIANT_SPLITROW:
      // the segment held on chip (one read) where it fits, else the streaming form
      if (!aligned) return SOFTMAX_ERR_MISALIGNED;
      if (splitrow_onchip_fits(p, dev)) {
        err = launch_splitrow_onchip_pooled(p, dev);
      } else {
        if (!splitrow_fits(p, dev)) return SOFTMAX_ERR_UNSUPPORTED;
        err = launch_splitrow(p, dev);
        variant = SOFTMAX_VARIANT_SPLITROW_STREAM;
      }
      break;
    case SOFTMAX_VARIANT_SPLITROW_STREAM:
      if (!aligned) return SOFTMAX_ERR_MISALIGNED;
      if (!splitrow_fits(p, dev)) return SOFTMAX_ERR_UNSUPPORTED;
      err = launch_splitrow(p, dev);
      break;
    default:
      return SOFTMAX_ERR_INVALID_ARG;
  }
  if (err != cudaSuccess) return cuda_fail(err);
  t_last_variant = variant;
  return SOFTMAX_OK;
}

// Many rows of 128 - 512 KiB and of 768 KiB - 1 MiB: a thread-block cluster per row, its CTAs'
// segments held on chip (measured against the cluster-row two passes, fp32: 4000 x 128 KiB 169
// against 182 us, 2000 x 256 KiB 168 / 193, 1000 x 512 KiB 161 / 196, 600 x 1 MiB 218 / 242; bf16
// 1000 x 512 KiB 167 / 206; ~1 GB per launch, TB/s: fp32 / bf16 896 KiB 5.83 / 5.48 against 5.54
// / 5.27, 1 MiB 5.84 / 5.42 against 5.46 / 5.24; but rows of 576 - 768 KiB, over clusters of 8,
// fp32 / bf16 576 KiB 4.58 / 4.69 against 5.62 / 5.09, 640 KiB 4.92 / 4.98 against 5.77 / 5.28,
// 768 KiB 5.44 / 5.42 against 5.68 / 5.22; 8000 x 80 KB 282 / 252 us, and fewer rows of 1 MiB,
// 100: 46.8 / 46.3, 20: 19.6 / 17.4).  Softmax and log softmax (contiguous rows, scale 1).
bool cluster_local_rows(const RowProblem& p, const DeviceInfo& dev) {
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  return row_bytes >= (int64_t(128) << 10) &&
         (row_bytes <= (int64_t(512) << 10)
              ? p.M >= int64_t(dev.sm_count)
              : row_bytes > (int64_t(768) << 10) && row_bytes <= (int64_t(1) << 20) && p.M >= 256) &&
         clusterrow_onchip_fits(p, dev);
}

// Row state only (optionally with the cross-entropy loss): the CTA bulk-copy kernel, whose copy
// ring keeps the next rows' reads in flight while a row is reduced, for aligned rows it holds;
// the two-pass kernel's first pass otherwise.
int run_state_only(RowProblem& p, const DeviceInfo& dev) {
  const bool aligned = aligned16(p.x) && (p.N * elem_bytes(p.dtype)) % 16 == 0;
  cudaError_t err;
  int variant;
  if (aligned && oneread_tma_fits(p, dev)) {
    err = launch_oneread_tma(p, dev);
    variant = SOFTMAX_VARIANT_ONEREAD_SMEM;
  } else {
    err = launch_twopass(p, aligned, dev);
    variant = SOFTMAX_VARIANT_TWOPASS;
  }
  if (err != cudaSuccess) return cuda_fail(err);
  t_last_variant = variant;
  return SOFTMAX_OK;
}

}  // namespace

int current_device(const DeviceInfo** out) { return current_device_info(out); }

int cuda_failure(cudaError_t err) { return cuda_fail(err); }

uint64_t local_wait_limit_ns() { return 2000ull * 1000 * 1000; }  // 2 s: never reached normally

uint64_t exchange_wait_limit_ns() {
  std::lock_guard<std::mutex> lock(g_debug_mutex);
  return g_exchange_wait_ns;
}

int debug_fault() {
  std::lock_guard<std::mutex> lock(g_debug_mutex);
  return g_debug_fault == 1 ? 1 : 0;
}

int debug_fault_attention() {
  std::lock_guard<std::mutex> lock(g_debug_mutex);
  return g_debug_fault == 2 ? 1 : 0;
}

}  // namespace rwo

using namespace rwo;

extern "C" {

int softmax_rows_ex(const void* x, void* y, float* m_out, float* d_out, float* lse_out, int64_t M,
                    int64_t N, int dtype, int variant, void* stream) {
  bool noop = false;
  int st = validate_rows(x, M, N, dtype, &noop);
  if (st != SOFTMAX_OK) return st;
  if (variant < SOFTMAX_VARIANT_AUTO || variant > SOFTMAX_VARIANT_SPLITROW_STREAM) return SOFTMAX_ERR_INVALID_ARG;
  if (noop) return SOFTMAX_OK;
  if (!y) return SOFTMAX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if ((st = current_device_info(&dev)) != SOFTMAX_OK) return st;
  RowProblem p;
  p.x = x;
  p.y = y;
  p.m_out = m_out;
  p.d_out = d_out;
  p.lse_out = lse_out;
  p.M = M;
  p.N = N;
  p.dtype = dtype;
  p.stream = static_cast<cudaStream_t>(stream);
  return run_variant(p, variant, *dev);
}

int softmax_rows(const void* x, void* y, int64_t M, int64_t N, int dtype, void* stream) {
  return softmax_rows_ex(x, y, nullptr, nullptr, nullptr, M, N, dtype, SOFTMAX_VARIANT_AUTO, stream);
}

int softmax_rows_causal(const void* x, void* y, float* m_out, float* d_out, float* lse_out, int64_t M, int64_t N,
                        int64_t q_period, int64_t key_offset, int dtype, void* stream) {
  bool noop = false;
  int st = validate_rows(x, M, N, dtype, &noop);
  if (st != SOFTMAX_OK) return st;
  if (q_period < 1) return SOFTMAX_ERR_INVALID_ARG;
  if (noop) return SOFTMAX_OK;
  if (!y) return SOFTMAX_ERR_INVALID_ARG;
  // Offsets beyond these bounds give the same lengths (all N, or all 0) and cannot overflow; a
  // period beyond M gives r % q_period = r for every row, as q_period = M does.
  if (q_period > M) q_period = M;
  if (key_offset > N) key_offset = N;
  if (key_offset < -q_period - 1) key_offset = -q_period - 1;
  const DeviceInfo* dev = nullptr;
  if ((st = current_device_info(&dev)) != SOFTMAX_OK) return st;
  RowProblem p;
  p.x = x;
  p.y = y;
  p.m_out = m_out;
  p.d_out = d_out;
  p.lse_out = lse_out;
  p.M = M;
  p.N = N;
  p.dtype = dtype;
  p.stream = static_cast<cudaStream_t>(stream);
  const bool aligned = aligned16(x) && aligned16(y) && (N * elem_bytes(dtype)) % 16 == 0;
  cudaError_t err;
  int variant;
  if (aligned && causal_warp_fits(p, *dev)) {  // rows up to 16 KiB: warp per row, live prefix only
    err = launch_causal_warp(p, *dev, q_period, key_offset);
    variant = SOFTMAX_VARIANT_ONEREAD_SMEM;
  } else {
    err = launch_twopass(p, aligned, *dev, q_period, key_offset);
    variant = SOFTMAX_VARIANT_TWOPASS;
  }
  if (err != cudaSuccess) return cuda_fail(err);
  t_last_variant = variant;
  return SOFTMAX_OK;
}

int softmax_rows_strided(const void* x, int64_t ldx, void* y, int64_t ldy, float* m_out, float* d_out,
                         float* lse_out, int64_t M, int64_t N, int dtype, float scale, int flags, int variant,
                         void* stream) {
  bool noop = false;
  int st = validate_rows(x, M, N, dtype, &noop);
  if (st != SOFTMAX_OK) return st;
  if (variant < SOFTMAX_VARIANT_AUTO || variant > SOFTMAX_VARIANT_SPLITROW_STREAM) return SOFTMAX_ERR_INVALID_ARG;
  if (flags & ~SOFTMAX_FLAG_LOG) return SOFTMAX_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale <= 3.4028234663852886e38f)) return SOFTMAX_ERR_INVALID_ARG;  // finite, > 0
  if (ldx == 0) ldx = N;
  if (ldy == 0) ldy = N;
  if (ldx < N || ldy < N) return SOFTMAX_ERR_INVALID_ARG;
  const int64_t s = elem_bytes(dtype);
  if (M > 0 && (ldx > INT64_MAX / s / M || ldy > INT64_MAX / s / M)) return SOFTMAX_ERR_INVALID_ARG;
  if (noop) return SOFTMAX_OK;
  if (!y) return SOFTMAX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if ((st = current_device_info(&dev)) != SOFTMAX_OK) return st;
  RowProblem p;
  p.x = x;
  p.y = y;
  p.m_out = m_out;
  p.d_out = d_out;
  p.lse_out = lse_out;
  p.M = M;
  p.N = N;
  p.dtype = dtype;
  p.log_out = (flags & SOFTMAX_FLAG_LOG) != 0;
  p.x_pitch = ldx * s;
  p.y_pitch = ldy * s;
  p.scale = scale;
  p.stream = static_cast<cudaStream_t>(stream);
  const int64_t row_bytes = N * s;
  const bool aligned = aligned16(x) && aligned16(y) && row_bytes % 16 == 0 && p.x_pitch % 16 == 0 &&
                       p.y_pitch % 16 == 0;
  if (variant == SOFTMAX_VARIANT_AUTO) {  // the kernels that take a pitch and a scale (and, for
                                          // contiguous rows at scale 1, the cluster kernel)
    if (aligned)
      variant = row_bytes <= (dtype == SOFTMAX_F32 ? 65536 : 8192) && oneread_reg_fits(p, true)
                    ? SOFTMAX_VARIANT_ONEREAD_REG
                : oneread_tma_fits(p, *dev) || cluster_local_rows(p, *dev) ? SOFTMAX_VARIANT_ONEREAD_SMEM
                                                                           : SOFTMAX_VARIANT_TWOPASS;
    else
      variant = (N <= 512 && oneread_reg_fits(p, false)) ? SOFTMAX_VARIANT_ONEREAD_REG : SOFTMAX_VARIANT_TWOPASS;
  }
  cudaError_t err;
  switch (variant) {
    case SOFTMAX_VARIANT_ONEREAD_REG:
      if (!oneread_reg_fits(p, aligned)) return SOFTMAX_ERR_UNSUPPORTED;
      err = launch_oneread_reg(p, aligned, *dev);
      break;
    case SOFTMAX_VARIANT_ONEREAD_SMEM:
      if (!aligned) return SOFTMAX_ERR_MISALIGNED;
      if (oneread_tma_fits(p, *dev))
        err = launch_oneread_tma(p, *dev);
      else if (clusterrow_onchip_fits(p, *dev))  // contiguous rows above the ring's reach, scale 1
        err = launch_clusterrow_onchip(p, *dev);
      else
        return SOFTMAX_ERR_UNSUPPORTED;
      break;
    case SOFTMAX_VARIANT_TWOPASS:
      err = launch_twopass_any(p, aligned, *dev);
      break;
    default:  // SOFTMAX_VARIANT_SPLITROW, SOFTMAX_VARIANT_SPLITROW_STREAM
      return SOFTMAX_ERR_UNSUPPORTED;
  }
  if (err != cudaSuccess) return cuda_fail(err);
  t_last_variant = variant;
  return SOFTMAX_OK;
}

int log_softmax_rows(const void* x, void* y, float* m_out, float* d_out, float* lse_out, int64_t M, int64_t N,
                     int dtype, int variant, void* stream) {
  return softmax_rows_strided(x, N, y, N, m_out, d_out, lse_out, M, N, dtype, 1.f, SOFTMAX_FLAG_LOG, variant,
                              stream);
}

int cross_entropy_rows(const void* x, const int64_t* labels, float* loss, float* lse_out, int64_t M, int64_t N,
                       int dtype, void* stream) {
  bool noop = false;
  int st = validate_rows(x, M, N, dtype, &noop);
  if (st != SOFTMAX_OK) return st;
  if (noop) return SOFTMAX_OK;
  if (!labels || !loss) return SOFTMAX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if ((st = current_device_info(&dev)) != SOFTMAX_OK) return st;
  RowProblem p;
  p.x = x;
  p.lse_out = lse_out;
  p.M = M;
  p.N = N;
  p.dtype = dtype;
  p.labels = labels;
  p.loss = loss;
  p.stream = static_cast<cudaStream_t>(stream);
  return run_state_only(p, *dev);
}

int attention_forward(const void* q, const void* k, const void* v, void* o, float* lse_out, int64_t BH, int64_t Sq,
                      int64_t Sk, int64_t d, float scale, int causal, int dtype, void* stream) {
  if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_BF16 && dtype != SOFTMAX_F16) return SOFTMAX_ERR_INVALID_ARG;
  if (BH < 0 || Sq < 1 || Sk < 1 || d < 1) return SOFTMAX_ERR_INVALID_ARG;
  if (scale == 0.f) scale = float(1.0 / sqrt(double(d)));  // the attention default, 1 / sqrt(d)
  if (!(scale > 0.f) || !(scale <= 3.4028234663852886e38f)) return SOFTMAX_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return SOFTMAX_ERR_INVALID_ARG;
  if (!attention_fits(d, dtype)) return SOFTMAX_ERR_UNSUPPORTED;
  // grid and copy-coordinate limits: BH indexes a grid dimension of at most 65535; rows are 32-bit
  // copy coordinates
  constexpr int64_t kMaxRows = (int64_t(1) << 31) - 256;
  if (BH > 65535 || Sq > kMaxRows || Sk > kMaxRows) return SOFTMAX_ERR_UNSUPPORTED;
  const int64_t row = d * elem_bytes(dtype);
  if (Sq > INT64_MAX / row / (BH > 0 ? BH : 1) || Sk > INT64_MAX / row / (BH > 0 ? BH : 1))
    return SOFTMAX_ERR_INVALID_ARG;
  if (BH == 0) return SOFTMAX_OK;
  if (!q || !k || !v || !o) return SOFTMAX_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return SOFTMAX_ERR_MISALIGNED;
  const DeviceInfo* dev = nullptr;
  int st = current_device_info(&dev);
  if (st != SOFTMAX_OK) return st;
  cudaError_t err = launch_attention(q, k, v, o, lse_out, BH, Sq, Sk, d, scale, causal != 0, dtype,
                                     static_cast<cudaStream_t>(stream), *dev);
  if (err != cudaSuccess) return cuda_fail(err);
  return SOFTMAX_OK;
}

int softmax_row_state(const void* x, float* m_out, float* d_out, float* lse_out, int64_t M, int64_t N,
                      int dtype, void* stream) {
  bool noop = false;
  int st = validate_rows(x, M, N, dtype, &noop);
  if (st != SOFTMAX_OK) return st;
  if (noop) return SOFTMAX_OK;
  if (!m_out && !d_out && !lse_out) return SOFTMAX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if ((st = current_device_info(&dev)) != SOFTMAX_OK) return st;
  RowProblem p;
  p.x = x;
  p.m_out = m_out;
  p.d_out = d_out;
  p.lse_out = lse_out;
  p.M = M;
  p.N = N;
  p.dtype = dtype;
  p.stream = static_cast<cudaStream_t>(stream);
  return run_state_only(p, *dev);
}

int merge_states(const float* m_a, const float* d_a, const float* m_b, const float* d_b, float* m_out,
                 float* d_out, float* lse_out, int64_t M, void* stream) {
  if (M < 0) return SOFTMAX_ERR_INVALID_ARG;
  if (M == 0) return SOFTMAX_OK;
  if (!m_a || !d_a || !m_b || !d_b || !m_out || !d_out) return SOFTMAX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  int st = current_device_info(&dev);
  if (st != SOFTMAX_OK) return st;
  cudaError_t err = launch_merge_states(m_a, d_a, m_b, d_b, m_out, d_out, lse_out, M,
                                        static_cast<cudaStream_t>(stream), *dev);
  if (err != cudaSuccess) return cuda_fail(err);
  return SOFTMAX_OK;
}

int softmax_rows_host(const void* x_host, void* y_host, int64_t M, int64_t N, int dtype, void* stream) {
  bool noop = false;
  int st = validate_rows(x_host, M, N, dtype, &noop);
  if (st != SOFTMAX_OK) return st;
  if (noop) return SOFTMAX_OK;
  if (!y_host) return SOFTMAX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  if ((st = current_device_info(&dev)) != SOFTMAX_OK) return st;

  const cudaStream_t user = static_cast<cudaStream_t>(stream);
  const int64_t row_bytes = N * elem_bytes(dtype);

  // Page-locked host buffers are directly addressable by the GPU (over NVLink-C2C on a
  // Grace-Blackwell node).  When both are, and the rows are at most 32 KiB (the register kernel's
  // range measured on this path), the register kernel reads x and writes y in host memory itself:
  // no staging copies, one pass over the link each way.  It uses plain loads and stores only.
  {
    void* dx = nullptr;
    void* dy = nullptr;
    if (cudaHostGetDevicePointer(&dx, const_cast<void*>(x_host), 0) == cudaSuccess &&
        cudaHostGetDevicePointer(&dy, y_host, 0) == cudaSuccess) {
      RowProblem p;
      p.x = dx;
      p.y = dy;
      p.M = M;
      p.N = N;
      p.dtype = dtype;
      p.stream = user;
      p.host_mem = true;
      const bool aligned = aligned16(dx) && aligned16(dy) && row_bytes % 16 == 0;
      if (row_bytes <= 32768 && oneread_reg_fits(p, aligned)) {
        cudaError_t err = launch_oneread_reg(p, aligned, *dev);
        if (err == cudaSuccess) err = cudaStreamSynchronize(user);
        if (err != cudaSuccess) return cuda_fail(err);
        t_last_variant = SOFTMAX_VARIANT_ONEREAD_REG;
        return SOFTMAX_OK;
      }
    } else {
      cudaGetLastError();  // pageable memory: not an error, take the staged path
    }
  }

  // Blocks of about 8 MiB: large enough for full-rate copies, small enough to overlap the
  // host->device copy of one block with the kernel and device->host copy of the others.
  int64_t block_rows = (int64_t(8) << 20) / row_bytes;
  if (block_rows < 1) block_rows = 1;
  if (block_rows > M) block_rows = M;
  const int64_t nblocks = (M + block_rows - 1) / block_rows;
  const size_t buf_bytes = size_t(block_rows * row_bytes);

  HostPipe& hp = g_pipe[dev->device];
  std::lock_guard<std::mutex> lock(hp.mu);
  cudaError_t err = hp.prepare(buf_bytes);
  if (err != cudaSuccess) return cuda_fail(err);

  int result = SOFTMAX_OK;
  auto fail = [&](cudaError_t e) {
    if (result == SOFTMAX_OK) result = cuda_fail(e);
  };
  if ((err = cudaEventRecord(hp.ev_start, user)) != cudaSuccess) return cuda_fail(err);
  for (int i = 0; i < HostPipe::kLanes; ++i)
    if ((err = cudaStreamWaitEvent(hp.lanes[i], hp.ev_start, 0)) != cudaSuccess) return cuda_fail(err);

  for (int64_t b = 0; b < nblocks; ++b) {
    const int li = int(b % HostPipe::kLanes);
    const int64_t r0 = b * block_rows;
    const int64_t rows = (M - r0) < block_rows ? (M - r0) : block_rows;
    const size_t bytes = size_t(rows * row_bytes);
    const char* src = static_cast<const char*>(x_host) + r0 * row_bytes;
    char* dst = static_cast<char*>(y_host) + r0 * row_bytes;
    if ((err = cudaMemcpyAsync(hp.buf[li], src, bytes, cudaMemcpyHostToDevice, hp.lanes[li])) != cudaSuccess) {
      fail(err);
      break;
    }
    RowProblem p;  // in place on the staging buffer
    p.x = hp.buf[li];
    p.y = hp.buf[li];
    p.M = rows;
    p.N = N;
    p.dtype = dtype;
    p.stream = hp.lanes[li];
    p.shares_gpu = true;  // the lanes' kernels overlap: none may need the whole GPU resident
    if ((st = run_variant(p, SOFTMAX_VARIANT_AUTO, *dev)) != SOFTMAX_OK) {
      result = st;
      break;
    }
    if ((err = cudaMemcpyAsync(dst, hp.buf[li], bytes, cudaMemcpyDeviceToHost, hp.lanes[li])) != cudaSuccess) {
      fail(err);
      break;
    }
  }
  // Join the lanes back into the caller's stream and wait for the result.
  for (int i = 0; i < HostPipe::kLanes; ++i) {
    if ((err = cudaEventRecord(hp.ev_done[i], hp.lanes[i])) != cudaSuccess) fail(err);
    else if ((err = cudaStreamWaitEvent(user, hp.ev_done[i], 0)) != cudaSuccess) fail(err);
  }
  if ((err = cudaStreamSynchronize(user)) != cudaSuccess) fail(err);
  return result;
}

int softmax_get_status(void* stream) {
  const DeviceInfo* dev = nullptr;
  int st = current_device_info(&dev);
  if (st != SOFTMAX_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned word = 0;
  cudaError_t err = cudaStreamSynchronize(s);
  if (err == cudaSuccess) err = cudaMemcpyAsync(&word, dev->status, sizeof word, cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess) err = cudaMemsetAsync(dev->status, 0, sizeof word, s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  if (err != cudaSuccess) return cuda_fail(err);
  if (word & kStatusTimeout) return SOFTMAX_ERR_TIMEOUT;
  if (word & kStatusBadLabel) return SOFTMAX_ERR_INVALID_ARG;
  return SOFTMAX_OK;
}

const char* softmax_status_string(int status) {
  switch (status) {
    case SOFTMAX_OK:
      return "ok";
    case SOFTMAX_ERR_INVALID_ARG:
      return "invalid argument";
    case SOFTMAX_ERR_MISALIGNED:
      return "pointer or row pitch not 16-byte aligned for the forced variant";
    case SOFTMAX_ERR_UNSUPPORTED:
      return "the forced variant cannot take this shape";
    case SOFTMAX_ERR_CUDA:
      return "CUDA error";
    case SOFTMAX_ERR_TIMEOUT:
      return "a kernel's bounded wait ran out";
    default:
      return "unknown status";
  }
}

const char* softmax_last_cuda_error(void) { return t_last_cuda_error.c_str(); }

int softmax_last_variant(void) { return t_last_variant; }

int softmax_debug_set_fault(int fault) {
  std::lock_guard<std::mutex> lock(g_debug_mutex);
  const int old = g_debug_fault;
  g_debug_fault = fault;
  return old;
}

int64_t softmax_debug_set_wait_limit_ns(int64_t ns) {
  std::lock_guard<std::mutex> lock(g_debug_mutex);
  const int64_t old = int64_t(g_exchange_wait_ns);
  if (ns > 0) g_exchange_wait_ns = uint64_t(ns);
  return old;
}

}  // extern "C"
