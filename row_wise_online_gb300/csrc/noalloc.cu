// noalloc.cu -- split-row softmax for callers that cannot allocate device memory.
//
// The regular split-row call (softmax_rows_ex with SOFTMAX_VARIANT_SPLITROW, or AUTO on few
// long rows) takes a small stream-ordered scratch buffer from the CUDA memory pool on every
// call: one 64-bit publication slot per (row, cluster) for the cross-cluster exchange.  Some
// callers cannot let a library allocate: code that must stay within a device-memory budget
// fixed up front, code whose framework allocator owns all device memory, and host threads
// that must not make a call that may block or synchronise the device.  This entry point makes
// the same kernel choice (each CTA's segment held on chip where it fits, else the streaming
// form) with its scratch in a file-scope device array instead, so it allocates nothing: no
// cudaMalloc / cudaMallocAsync / cudaFree, no library allocator.
#include <mutex>

#include "../../include/softmax_rows.h"
#include "launch.h"

namespace rwo {
namespace {

// 40960 slots of 8 bytes = 320 KiB, resident on every device that loads the library until the
// process exits.  A call needs M x (number of clusters) slots.
constexpr size_t kNoAllocSlots = 40960;
static __device__ __align__(256) unsigned long long g_noalloc_pub[kNoAllocSlots];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
unsigned long long* g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_pub, per device

// Set-up on the first call on a device (with that device current): in host code the array's
// name is only a host-side stand-in, so its device address is looked up once and kept.
cudaError_t noalloc_scratch(int device, unsigned long long** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[device]) {
    void* ptr = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&ptr, g_noalloc_pub);
    if (err != cudaSuccess) return err;
    g_noalloc_ptr[device] = static_cast<unsigned long long*>(ptr);
  }
  *out = g_noalloc_ptr[device];
  return cudaSuccess;
}

}  // namespace
}  // namespace rwo

using namespace rwo;

extern "C" int softmax_rows_splitrow_noalloc(const void* x, void* y, float* m_out, float* d_out, float* lse_out,
                                             int64_t M, int64_t N, int dtype, void* stream) {
  if (dtype != SOFTMAX_F32 && dtype != SOFTMAX_BF16 && dtype != SOFTMAX_F16) return SOFTMAX_ERR_INVALID_ARG;
  if (N < 1 || M < 0) return SOFTMAX_ERR_INVALID_ARG;
  const int64_t s = elem_bytes(dtype);
  if (N > INT64_MAX / s) return SOFTMAX_ERR_INVALID_ARG;
  if (M == 0) return SOFTMAX_OK;
  if (M > INT64_MAX / (N * s)) return SOFTMAX_ERR_INVALID_ARG;
  if (!x || !y) return SOFTMAX_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(y) & 15u) || (N * s) % 16)
    return SOFTMAX_ERR_MISALIGNED;
  const DeviceInfo* dev = nullptr;
  const int st = current_device(&dev);
  if (st != SOFTMAX_OK) return st;
  if (dev->device < 0 || dev->device >= kMaxDevices) return SOFTMAX_ERR_UNSUPPORTED;
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
  // the same kernel choice as SOFTMAX_VARIANT_SPLITROW: the segment held on chip where it fits
  const bool onchip = splitrow_onchip_fits(p, *dev);
  if (!onchip && !splitrow_fits(p, *dev)) return SOFTMAX_ERR_UNSUPPORTED;
  const size_t slots = onchip ? size_t(M) * size_t(splitrow_onchip_clusters(p, *dev)) : splitrow_slots(p, *dev);
  if (slots > kNoAllocSlots) return SOFTMAX_ERR_UNSUPPORTED;
  unsigned long long* pub = nullptr;
  cudaError_t err = noalloc_scratch(dev->device, &pub);
  if (err != cudaSuccess) return cuda_failure(err);
  if (onchip) {
    // the slots must read as "not published" (all ones) when the kernel starts
    err = cudaMemsetAsync(pub, 0xFF, slots * sizeof(unsigned long long), p.stream);
    if (err == cudaSuccess) err = launch_splitrow_onchip(p, *dev, pub);
  } else {
    bool too_big = false;
    err = launch_splitrow_scratch(p, *dev, pub, kNoAllocSlots, &too_big);
    if (too_big) return SOFTMAX_ERR_UNSUPPORTED;
  }
  if (err != cudaSuccess) return cuda_failure(err);
  return SOFTMAX_OK;
}
