// kernel_clusterrow.cu -- long rows at many rows: one thread-block cluster per row, two passes.
//
// "5.2 CUDA Online Softmax 实现优化" §7.1 names the case of rows too long for one block (split a
// row over several blocks and merge their partial (m, d) results); the merge is the (m, d) merge
// of §4.1, associative, so any partition of a row can be folded separately and combined.
//
// Why clusters rather than a CTA per row: a two-pass CTA per row keeps (resident CTAs) x (row
// bytes) in flight, which passes the size of L2 once rows reach a few hundred KiB -- the second
// read of a row then comes from HBM again and the kernel moves three row-lengths per row instead
// of two (measured: ~4.4 TB/s for 1-8 MiB fp32 rows).  Here a cluster of CS CTAs shares each row,
// so only (resident CTAs / CS) rows are in flight; the host picks CS so that they fit in L2 (CS =
// 1, a CTA per row, up to rows of ~260 KiB)
// (measured, fp32, against a CTA per row: 512 KiB rows 4.75 -> 5.17 TB/s, 1 MiB 4.45 -> 5.09,
// 2 MiB 4.30 -> 5.13, 4 MiB 4.47 -> 4.96).
//
// Per row, in every CTA of the cluster (rank q of CS):
//   1. pass 1 over the CTA's contiguous segment q of the row's 16-byte units: each thread folds
//      its units with the online update (the step maximum first, one exponential per element,
//      one rescale of the running sum per step, compensated sum); loads marked L2::evict_last;
//   2. warp butterfly + cross-warp merge -> the CTA state, written to this CTA's shared memory;
//   3. cluster barrier; warp 0 reads the CS CTA states over distributed shared memory (lane i
//      reads rank i) and merges them with the warp butterfly -- the same inputs and the same
//      steps in every CTA, so every CTA normalises with bitwise the same (m, d);
//   4. pass 2 over the segment: y = e^(x - m) / d (or the log form), re-read from L2 (loads
//      marked evict_first), 16-byte streaming stores; from the segment's end when the rows in
//      flight come near the size of L2.
// The clusters walk the rows with a stride of the cluster count.  A cluster barrier is a
// hardware barrier over CTAs that are co-scheduled by construction (a cluster launches whole),
// so it needs no time limit.
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

constexpr int kCrUnroll = 4;               // 16-byte units per thread per step
constexpr int kCrThreads = 512;            // threads per CTA (two CTAs per SM)
// Rows in flight x row bytes stays below this (measured, fp32 rows of 512 KiB - 2 MiB: 76 MB in
// flight with the smaller cluster beat 38 MB with the next larger one by 2-9%; the clusters of 16
// that 4 MiB rows need run slower than those of 8).
constexpr int64_t kCrInflightBytes = 80ll << 20;
constexpr int64_t kCrReverseBytes = 64ll << 20;  // rows in flight above this: pass 2 runs backwards

struct ClusterRowArgs {
  const unsigned char* x;
  unsigned char* y;
  float* m_out;
  float* d_out;
  float* lse_out;
  int64_t M;
  int64_t units;  // 16-byte units per row
  int64_t x_pitch, y_pitch;  // bytes between rows
  float scale;               // softmax of scale * x
  float c;                   // scale * log2 e
  int p2_reverse;            // pass 2 walks the segment from its end
};

__device__ __forceinline__ uint32_t cr_cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// 16-byte load with an L2 eviction policy (no L1 allocation).
__device__ __forceinline__ uint4 ld16_policy(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

__device__ __forceinline__ State ld_cluster_state(uint32_t addr) {
  State s;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(s.m), "=f"(s.d) : "r"(addr) : "memory");
  return s;
}

template <class D, bool LOG>
__global__ void __launch_bounds__(kCrThreads, 2) k_clusterrow(ClusterRowArgs a) {
  constexpr int E = D::kVec;
  constexpr int U = kCrUnroll;
  constexpr int nt = kCrThreads;  // launched with exactly this many threads
  __shared__ State slots[2][kCrThreads / 32];
  __shared__ __align__(8) State cta_state[2];  // this CTA's state of the row, by row parity
  __shared__ State row_state[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t cs = cr_cluster_size();
  const int64_t ncl = cluster_count_x();
  // this CTA's segment of every row: the units cut in cs contiguous near-equal parts
  const int64_t per = a.units / cs, rem = a.units % cs;
  const int64_t u0 = int64_t(rank) * per + (int64_t(rank) < rem ? rank : rem);
  const int64_t nu = per + (int64_t(rank) < rem ? 1 : 0);
  const uint64_t keep = policy_evict_last(), drop = policy_evict_first();

  int it = 0;
  for (int64_t row = cluster_id_x(); row < a.M; row += ncl, ++it) {
    const unsigned char* xs = a.x + row * a.x_pitch + u0 * 16;
    // pass 1: online fold of the segment, one rescale per step of U units, compensated sum
    float m = -INFINITY, d = 0.f, c = 0.f;
    for (int64_t base = threadIdx.x; base < nu; base += int64_t(nt) * U) {
      const int64_t left = nu - base;  // units of this thread's step k exist while k * nt < left
      const unsigned char* xp = xs + base * 16;
      uint4 q[U];  // raw vectors: the loads of a step are all in flight before the first use
#pragma unroll
      for (int k = 0; k < U; ++k)
        if (int64_t(k) * nt < left) q[k] = ld16_policy(xp + k * nt * 16, keep);
      float mu = -INFINITY;
#pragma unroll
      for (int k = 0; k < U; ++k)
        if (int64_t(k) * nt < left) mu = fmaxf(mu, D::vmax(q[k]));
      const float m_new = fmaxf(m, mu);
      const float ms = safe_max(m_new);
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < U; ++k) {
        if (int64_t(k) * nt < left) {
          float v[E];
          D::unpack(q[k], v);
#pragma unroll
          for (int e = 0; e < E; ++e) acc += exp_diff(v[e], ms, a.c);
        }
      }
      const float r = exp_diff(m, ms, a.c);  // rescale of the running sum; 0 when m was -inf
      const float ds = __fmul_rn(d, r);
      c = __fmul_rn(c, r);
      const float yk = __fsub_rn(acc, c);
      const float t = __fadd_rn(ds, yk);
      c = __fsub_rn(__fsub_rn(t, ds), yk);
      d = t;
      m = m_new;
    }
    const State s_cta = group_merge(State{m, d}, slots[it & 1], nt >> 5, warp, lane, [] { __syncthreads(); }, a.c);
    if (threadIdx.x == 0) cta_state[it & 1] = s_cta;
    // Every CTA's state of this row is visible to the cluster.  The buffer written here is
    // written again two rows later, after the next row's barrier, which every CTA reaches only
    // after its reads below.
    cluster_sync();
    if (warp == 0) {
      State t = empty_state();
      if (uint32_t(lane) < cs) t = ld_cluster_state(map_to_rank(smem_addr(&cta_state[it & 1]), lane));
      t = warp_merge(t, a.c);  // lanes past cs hold the empty state, the merge identity
      if (lane == 0) row_state[it & 1] = t;
    }
    __syncthreads();
    const State s = row_state[it & 1];
    // pass 2: re-read (from L2) and normalise
    const float ms = safe_max(s.m);
    const float inv = safe_inv(s.d);
    const LogNorm ln = log_norm(s);
    unsigned char* ys = a.y + row * a.y_pitch + u0 * 16;
    // When the rows in flight come near the size of L2, the last step first: the lines read
    // last in pass 1 are the likeliest to be still there (measured on fp32 rows of 512 KiB -
    // 6 MiB with ~76 MB or more in flight: +1.3-2.4%; with ~57 MB in flight it costs ~1%).
    const int64_t nsteps = threadIdx.x < nu ? (nu - threadIdx.x + int64_t(nt) * U - 1) / (int64_t(nt) * U) : 0;
    for (int64_t j = 0; j < nsteps; ++j) {
      const int64_t base = threadIdx.x + (a.p2_reverse ? nsteps - 1 - j : j) * int64_t(nt) * U;
      const int64_t left = nu - base;
      const unsigned char* xp = xs + base * 16;
      unsigned char* yp = ys + base * 16;
      uint4 q[U];
#pragma unroll
      for (int k = 0; k < U; ++k)
        if (int64_t(k) * nt < left) q[k] = ld16_policy(xp + k * nt * 16, drop);
#pragma unroll
      for (int k = 0; k < U; ++k) {
        if (int64_t(k) * nt < left) {
          float v[E];
          D::unpack(q[k], v);
#pragma unroll
          for (int e = 0; e < E; ++e)
            v[e] = LOG ? log_prob(v[e], ln, a.scale) : __fmul_rn(exp_diff(v[e], ms, a.c), inv);
          st_stream16(yp + k * nt * 16, D::pack(v));
        }
      }
    }
    if (rank == 0 && threadIdx.x == 0) {
      const State o = scaled_state(s, a.scale);
      if (a.m_out) a.m_out[row] = o.m;
      if (a.d_out) a.d_out[row] = o.d;
      if (a.lse_out) a.lse_out[row] = lse_of(o);
    }
  }
  // no CTA leaves while another CTA of the cluster may still read its shared memory
  cluster_sync();
}

using ClusterRowKernel = void (*)(ClusterRowArgs);

ClusterRowKernel clusterrow_kernel(int dtype, bool log) {
  static const ClusterRowKernel table[3][2] = {{k_clusterrow<F32, false>, k_clusterrow<F32, true>},
                                               {k_clusterrow<BF16, false>, k_clusterrow<BF16, true>},
                                               {k_clusterrow<F16, false>, k_clusterrow<F16, true>}};
  return table[dtype][log ? 1 : 0];
}

struct ClusterRowPlan {
  int cluster = 0;   // CTAs per cluster (0: the kernel does not take the problem)
  int clusters = 0;  // resident clusters launched
};

int max_active_clusters(ClusterRowKernel fn, int cs) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(kCrThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (const void*)fn, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

constexpr int kCrSizes[5] = {1, 2, 4, 8, 16};

// Resident clusters of each size, per device and kernel: queried once (the occupancy queries
// cost far more than a launch).
struct ResidentClusters {
  int n[5] = {0, 0, 0, 0, 0};
};
std::mutex g_cr_mutex;
ResidentClusters g_cr[64][3][2];
bool g_cr_ready[64][3][2];

ResidentClusters resident_clusters(int dtype, bool log, const DeviceInfo& dev) {
  std::lock_guard<std::mutex> lock(g_cr_mutex);
  const bool cache = dev.device >= 0 && dev.device < 64;
  if (cache && g_cr_ready[dev.device][dtype][log]) return g_cr[dev.device][dtype][log];
  ResidentClusters r;
  ClusterRowKernel fn = clusterrow_kernel(dtype, log);
  if (cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    cudaGetLastError();  // clusters of 16 then report no residency
  for (int i = 0; i < 5; ++i) r.n[i] = max_active_clusters(fn, kCrSizes[i]);
  if (cache) {
    g_cr[dev.device][dtype][log] = r;
    g_cr_ready[dev.device][dtype][log] = true;
  }
  return r;
}

// The smallest cluster (1 .. 16 CTAs) whose resident clusters keep at most kCrInflightBytes of
// rows in flight; the largest one when none does.  A cluster of one CTA is a CTA per row, at two
// CTAs of 512 threads per SM and with the L2 hints (measured against the 1024-thread two-pass
// kernel, rows of 128-192 KiB: fp32 5.1-5.3 -> 5.7-5.9 TB/s, bf16 4.6-5.0 -> 5.3-5.5).
ClusterRowPlan plan_clusterrow(const RowProblem& p, const DeviceInfo& dev) {
  ClusterRowPlan plan;
  if (!dev.cluster_launch) return plan;
  const ResidentClusters r = resident_clusters(p.dtype, p.log_out, dev);
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  for (int i = 0; i < 5; ++i) {
    if (r.n[i] < 1) continue;
    plan.cluster = kCrSizes[i];
    plan.clusters = r.n[i];
    if (int64_t(r.n[i]) * row_bytes <= kCrInflightBytes) break;
  }
  return plan;
}

}  // namespace

bool clusterrow_fits(const RowProblem& p, const DeviceInfo& dev) {
  if (p.y == nullptr || p.labels || p.loss) return false;
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  if (row_bytes % 16 != 0) return false;
  if ((p.x_pitch % 16) != 0 || (p.y_pitch % 16) != 0) return false;
  return plan_clusterrow(p, dev).cluster > 0;
}

cudaError_t launch_clusterrow(const RowProblem& p, const DeviceInfo& dev) {
  const ClusterRowPlan plan = plan_clusterrow(p, dev);
  if (plan.cluster == 0) return cudaErrorInvalidConfiguration;
  ClusterRowKernel fn = clusterrow_kernel(p.dtype, p.log_out);
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  ClusterRowArgs a;
  a.x = static_cast<const unsigned char*>(p.x);
  a.y = static_cast<unsigned char*>(p.y);
  a.m_out = p.m_out;
  a.d_out = p.d_out;
  a.lse_out = p.lse_out;
  a.M = p.M;
  a.units = row_bytes / 16;
  a.x_pitch = p.x_pitch ? p.x_pitch : row_bytes;
  a.y_pitch = p.y_pitch ? p.y_pitch : row_bytes;
  a.scale = p.scale;
  a.c = p.scale * kLog2e;
  const int64_t clusters = p.M < plan.clusters ? p.M : plan.clusters;
  a.p2_reverse = clusters * row_bytes > kCrReverseBytes ? 1 : 0;

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(unsigned(clusters * plan.cluster));
  cfg.blockDim = dim3(kCrThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = p.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace rwo
