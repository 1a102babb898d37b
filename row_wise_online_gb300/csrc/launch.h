// launch.h -- internal interface between the C ABI (api.cu) and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rwo {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int max_smem_per_block_optin = 0;  // bytes of dynamic + static shared memory a block may use
  int max_smem_per_sm = 0;
  int max_threads_per_sm = 0;
  int l2_bytes = 0;
  int cluster_launch = 0;
  unsigned* status = nullptr;  // device address of this device's status word
};

// One softmax problem.  Pointers are device pointers; y may be null for state-only work.
struct RowProblem {
  const void* x = nullptr;
  void* y = nullptr;
  float* m_out = nullptr;
  float* d_out = nullptr;
  float* lse_out = nullptr;
  int64_t M = 0;
  int64_t N = 0;
  int dtype = 0;  // 0 = fp32, 1 = bf16, 2 = fp16
  bool log_out = false;  // y = log-softmax instead of softmax (register, CTA bulk-copy, two-pass)
  const int64_t* labels = nullptr;  // cross entropy (two-pass, no y): loss[r] = LSE_r - x_r[labels[r]]
  float* loss = nullptr;
  int64_t x_pitch = 0, y_pitch = 0;  // bytes between rows (0: N * element size); register, CTA
  float scale = 1.f;                 // bulk-copy and two-pass kernels: softmax of scale * x
  cudaStream_t stream = nullptr;
  bool host_mem = false;  // x and y are page-locked host memory read and written over the host link
  bool shares_gpu = false;  // other kernels may run beside this launch (the split-row kernel is then off)
};

// Status bits a kernel may set in the per-device status word.
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBadLabel = 2u;  // a cross-entropy label >= N

inline int elem_bytes(int dtype) { return dtype == 0 ? 4 : 2; }

// Host-side wait limits handed to kernels (nanoseconds).
uint64_t local_wait_limit_ns();     // waits on this CTA's own copies and threads
uint64_t exchange_wait_limit_ns();  // waits on other clusters (split row)
int debug_fault();                  // test hook (split row): 1 = cluster 0 never publishes
int debug_fault_attention();        // test hook (attention): 2 = the first V tile is never copied

// Each `*_fits` says whether the variant can take the problem (alignment already checked by
// the caller where the variant needs it).  Each `launch_*` enqueues the work and returns a
// cudaError_t from the launch.
bool oneread_reg_fits(const RowProblem& p, bool vec);
cudaError_t launch_oneread_reg(const RowProblem& p, bool vec, const DeviceInfo& dev);

bool oneread_warp_fits(const RowProblem& p, const DeviceInfo& dev);
cudaError_t launch_oneread_warp(const RowProblem& p, const DeviceInfo& dev);

// Causal rows (q_period >= 1): row r keeps its first clamp(r % q_period + 1 + key_offset, 0, N)
// entries; the rest are not read and give y = 0.
bool causal_warp_fits(const RowProblem& p, const DeviceInfo& dev);
cudaError_t launch_causal_warp(const RowProblem& p, const DeviceInfo& dev, int64_t q_period, int64_t key_offset);

bool oneread_tma_fits(const RowProblem& p, const DeviceInfo& dev);
cudaError_t launch_oneread_tma(const RowProblem& p, const DeviceInfo& dev);

// q_period >= 1 applies the causal rule above; 0 processes whole rows.
cudaError_t launch_twopass(const RowProblem& p, bool vec, const DeviceInfo& dev, int64_t q_period = 0,
                           int64_t key_offset = 0);

// Two passes with a thread-block cluster per row (16-byte aligned rows and pitches, y written,
// no cross entropy); for long rows at many rows, where a CTA per row would keep more rows in
// flight than L2 holds.
bool clusterrow_fits(const RowProblem& p, const DeviceInfo& dev);
cudaError_t launch_clusterrow(const RowProblem& p, const DeviceInfo& dev);

bool splitrow_fits(const RowProblem& p, const DeviceInfo& dev);
cudaError_t launch_splitrow(const RowProblem& p, const DeviceInfo& dev);

// Split row with each CTA's segment held in shared memory (one read of x): 16-byte aligned rows
// whose per-CTA segment fits at least two row buffers.  `pub` holds M x splitrow_onchip_clusters()
// 64-bit publication slots, all ones when the kernel starts (the _pooled form allocates and sets
// them on the stream).
bool splitrow_onchip_fits(const RowProblem& p, const DeviceInfo& dev);
int splitrow_onchip_clusters(const RowProblem& p, const DeviceInfo& dev);
cudaError_t launch_splitrow_onchip(const RowProblem& p, const DeviceInfo& dev, unsigned long long* pub);
cudaError_t launch_splitrow_onchip_pooled(const RowProblem& p, const DeviceInfo& dev);
// The same kernel with each thread-block cluster owning whole rows (rows k, k + clusters, ... for
// cluster k; 16-byte aligned contiguous rows, y written, softmax without scale): the row's CTA states
// merged over DSMEM only.  For many long rows (~256 KiB - 2 MiB).
bool clusterrow_onchip_fits(const RowProblem& p, const DeviceInfo& dev);
cudaError_t launch_clusterrow_onchip(const RowProblem& p, const DeviceInfo& dev);
// Publication slots the streaming split-row kernel needs (M x its clusters).
size_t splitrow_slots(const RowProblem& p, const DeviceInfo& dev);

// Split row with caller-provided scratch: `pub` holds `pub_slots` 64-bit publication slots
// (device memory).  Nothing is allocated.  Returns cudaErrorInvalidValue when the problem
// needs more slots than given (*too_big is then set).
cudaError_t launch_splitrow_scratch(const RowProblem& p, const DeviceInfo& dev, unsigned long long* pub,
                                    size_t pub_slots, bool* too_big);

// The current device's properties (softmax_status code), for entry points outside api.cu.
int current_device(const DeviceInfo** out);
// Records err as the thread's last CUDA error and returns SOFTMAX_ERR_CUDA.
int cuda_failure(cudaError_t err);

cudaError_t launch_merge_states(const float* m_a, const float* d_a, const float* m_b,
                                const float* d_b, float* m_out, float* d_out, float* lse_out,
                                int64_t M, cudaStream_t stream, const DeviceInfo& dev);

}  // namespace rwo
