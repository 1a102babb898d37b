// kernel_splitrow.cu -- split-row softmax: few, very long rows spread over the whole GPU.
//
// "5.2 CUDA Online Softmax 实现优化" §7.1 names the case (small M, huge N: split one row over
// several blocks and merge their partial results); the merge is the (m, d) merge of §4.1, which
// is associative, so any partition of a row can be folded separately and combined.
//
// Layout: the grid is G persistent CTAs (one per SM), grouped in thread-block clusters of CS.
// Every row is cut into G contiguous segments of 16-byte units, balanced to one unit; CTA c owns
// segment c of every row.  One producer lane streams the segments of consecutive rows, in 15 KB
// pieces, through a ring of shared-memory slots with bulk copies (cp.async.bulk + mbarrier).
// Consumers copy each piece into registers as soon as it lands and free its slot, so the ring
// only ever holds loads in flight and HBM reads keep streaming while a row waits for its
// exchange.  x is read once; y is written once, straight from registers.
//
// Per row r, in every CTA:
//   1. consumers gather the segment (up to 8 pieces, 2 vectors per thread per piece)
//      into registers, take the thread max, then one exponential per element: the thread's
//      (m, d) state;
//   2. warp butterfly merge, then cross-warp merge through shared memory -> CTA state;
//   3. cluster merge over distributed shared memory: each CTA writes its state into rank 0's
//      shared memory (st.shared::cluster) and arrives on rank 0's mbarrier (release.cluster);
//      rank 0 merges the CS states in rank order and publishes the cluster state to global
//      memory, then bumps a release counter;
//   4. one lane waits (acquire, bounded by %globaltimer) until every cluster has published row
//      r; warp 0 merges all cluster states in a fixed order -- identical in every CTA, so every
//      CTA normalises with bitwise the same (m, d);
//   5. y = e^(x - m) / d from registers, 16-byte stores.
// All clusters must be resident at once; the host launches at most the number of clusters the
// occupancy query reports.  Every wait is bounded; a wait that runs out records
// SOFTMAX_ERR_TIMEOUT in the status word, skips the remaining exchange waits, and the kernel
// still terminates.
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

// 15 consumer warps + 1 producer warp = 16 warps, 4 per SM sub-partition, so each thread may
// use up to 128 registers (17 warps would cap it at 96 and spill the row).
constexpr int kSplitNcw = 15;                                    // consumer warps
constexpr int kSplitNct = kSplitNcw * 32;                        // consumer threads
constexpr int kUnitsPerPiecePerThread = 2;
constexpr int kPieceUnits = kSplitNct * kUnitsPerPiecePerThread;  // 960 units
constexpr int kPieceBytes = kPieceUnits * 16;                    // 15 KB
// Register capacity per CTA and row: 8 pieces (120 KB) for fp32; 6 for bf16, whose unpacking
// needs more temporaries (7 or 8 would spill).
template <class D>
__host__ __device__ constexpr int max_pieces() { return D::kBytes == 4 ? 8 : 6; }
constexpr int kMaxCluster = 8;
static_assert(kPieceUnits % kSplitNct == 0, "a piece splits evenly over the consumer threads");

struct SplitArgs {
  const unsigned char* x;
  unsigned char* y;
  float* m_out;
  float* d_out;
  float* lse_out;
  int64_t M;
  int64_t units;  // 16-byte units per row
  int64_t row_bytes;
  int slots;          // ring slots of kPieceBytes
  unsigned* counter;  // cluster publications so far (zeroed before launch)
  float* gstate;      // [M][clusters][2]: published cluster states
  unsigned* status;
  uint64_t local_wait_ns;
  uint64_t exchange_wait_ns;
  int fault;  // test hook: cluster 0 never publishes
};

size_t split_tail_bytes(int slots) {
  return size_t(slots) * 2 * sizeof(uint64_t) + 2 * sizeof(uint64_t) + 2 * kMaxCluster * sizeof(State) +
         2 * kSplitNcw * sizeof(State) + 2 * sizeof(State) + 16;
}

__device__ __forceinline__ float ld_relaxed_f32(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync_all() {
  // Non-aligned form: the producer warp's lanes reach it from different paths.
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

template <class D>
__global__ void __launch_bounds__((kSplitNcw + 1) * 32, 1) k_splitrow(SplitArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int E = D::kVec;
  constexpr int U = kUnitsPerPiecePerThread;
  constexpr int KMAX = max_pieces<D>();
  const int NS = a.slots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(NS) * kPieceBytes);
  uint64_t* freed = full + NS;
  uint64_t* cbar = freed + NS;                                // [2]
  State* cstate = reinterpret_cast<State*>(cbar + 2);        // [2][kMaxCluster], written into rank 0
  State* wstate = cstate + 2 * kMaxCluster;                  // [2][kSplitNcw]
  State* rowst = wstate + 2 * kSplitNcw;                     // [2]
  int* abort_flag = reinterpret_cast<int*>(rowst + 2);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const uint32_t cid = cluster_id_x();
  const uint32_t ncl = cluster_count_x();

  // This CTA's segment of every row, in 16-byte units.
  const int64_t G = gridDim.x, c = blockIdx.x;
  const int64_t base = a.units / G, rem = a.units % G;
  const int64_t seg_units = base + (c < rem ? 1 : 0);
  const int64_t seg_start = c * base + (c < rem ? c : rem);
  const int K = int((seg_units + kPieceUnits - 1) / kPieceUnits);  // <= KMAX (the host checks)

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&freed[s]), kSplitNcw);
    }
    mbar_init(smem_addr(&cbar[0]), csize);
    mbar_init(smem_addr(&cbar[1]), csize);
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive

  if (warp == kSplitNcw) {
    // ---------------- producer: stream pieces of consecutive rows through the ring ----------------
    if (lane == 0 && K > 0) {
      const uint64_t pol = policy_evict_first();
      const int64_t total = a.M * K;
      bool timed_out = false;
      for (int64_t p = 0; p < total; ++p) {
        const int s = int(p % NS);
        if (p >= NS &&
            !mbar_wait(smem_addr(&freed[s]), uint32_t(((p / NS) - 1) & 1), a.local_wait_ns))
          timed_out = true;
        const int64_t r = p / K;
        const int k = int(p % K);
        const int64_t rest = seg_units - int64_t(k) * kPieceUnits;
        const uint32_t bytes = uint32_t(rest < kPieceUnits ? rest : kPieceUnits) * 16u;
        const uint32_t bar = smem_addr(&full[s]);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(smem_addr(smem + size_t(s) * kPieceBytes),
                 a.x + r * a.row_bytes + (seg_start + int64_t(k) * kPieceUnits) * 16, bytes, bar, pol);
      }
      // every load has landed before the CTA may exit (the consumers normally saw them all)
      for (int64_t p = total > NS ? total - NS : 0; p < total; ++p)
        if (!mbar_wait(smem_addr(&full[p % NS]), uint32_t((p / NS) & 1), a.local_wait_ns)) timed_out = true;
      if (timed_out) atomicOr(a.status, kStatusTimeout);
    }
  } else {
    // ---------------- consumers ----------------
    bool timed_out = false;
    for (int64_t r = 0; r < a.M; ++r) {
      const int b = int(r & 1);
      // 1. gather the segment into registers, freeing each slot at once
      uint4 v[KMAX][U];
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
#pragma unroll
        for (int i = 0; i < U; ++i) v[k][i] = make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
        if (k < K) {
          const int64_t p = r * K + k;
          const int s = int(p % NS);
          if (!mbar_wait(smem_addr(&full[s]), uint32_t((p / NS) & 1), a.local_wait_ns)) timed_out = true;
          const uint32_t slot = smem_addr(smem + size_t(s) * kPieceBytes);
          const int64_t rest = seg_units - int64_t(k) * kPieceUnits;
#pragma unroll
          for (int i = 0; i < U; ++i) {
            const int u = tid + i * kSplitNct;
            if (u < rest) v[k][i] = lds16(slot + uint32_t(u) * 16u);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&freed[s]));
        }
      }
      // thread state: max first, then one exponential per element
      float mt = -INFINITY;
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
#pragma unroll
        for (int i = 0; i < U; ++i) mt = fmaxf(mt, D::vmax(v[k][i]));
      const float mts = safe_max(mt);
      float dt = 0.f;
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
#pragma unroll
        for (int i = 0; i < U; ++i) {
          float f[E];
          D::unpack(v[k][i], f);
#pragma unroll
          for (int e = 0; e < E; ++e) dt += exp_diff(f[e], mts);
        }
      // 2. CTA merge
      const State st = group_merge(State{mt, dt}, wstate + b * kSplitNcw, kSplitNcw, warp, lane,
                                   [] { named_barrier_sync(1, kSplitNct); });
      // 3. cluster merge over DSMEM; rank 0 publishes the cluster state
      if (tid == 0) {
        st_cluster_f32x2(map_to_rank(smem_addr(&cstate[b * kMaxCluster + crank]), 0), st.m, st.d);
        mbar_arrive_remote(map_to_rank(smem_addr(&cbar[b]), 0));
        if (crank == 0) {
          if (!mbar_wait_cluster(smem_addr(&cbar[b]), uint32_t((r >> 1) & 1), a.local_wait_ns)) timed_out = true;
          State cs = empty_state();
          for (uint32_t i = 0; i < csize; ++i) cs = merge(cs, cstate[b * kMaxCluster + i]);
          if (!(a.fault && cid == 0)) {
            float* g = a.gstate + (r * ncl + cid) * 2;
            g[0] = cs.m;
            g[1] = cs.d;
            red_release_add(a.counter, 1u);
          }
        }
      }
      // 4. wait for every cluster's state of row r, then merge them in cluster order
      if (warp == 0) {
        if (lane == 0 && *abort_flag == 0) {
          const unsigned target = unsigned((r + 1) * ncl);
          if (ld_acquire(a.counter) < target) {
            const uint64_t t0 = global_timer_ns();
            while (ld_acquire(a.counter) < target) {
              if (global_timer_ns() - t0 > a.exchange_wait_ns) {
                *abort_flag = 1;
                timed_out = true;
                break;
              }
              __nanosleep(32);
            }
          }
        }
        __syncwarp();
        State g = empty_state();
        for (uint32_t i = lane; i < ncl; i += 32) {
          const float* gp = a.gstate + (r * ncl + i) * 2;
          g = merge(g, State{ld_relaxed_f32(gp), ld_relaxed_f32(gp + 1)});
        }
        g = warp_merge(g);
        if (lane == 0) rowst[b] = g;
      }
      named_barrier_sync(1, kSplitNct);
      const State row = rowst[b];
      // 5. normalise from registers and store
      const float ms = safe_max(row.m);
      const float inv = safe_inv(row.d);
      unsigned char* yseg = a.y + r * a.row_bytes + seg_start * 16;
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
        if (k < K) {
          const int64_t rest = seg_units - int64_t(k) * kPieceUnits;
#pragma unroll
          for (int i = 0; i < U; ++i) {
            const int u = tid + i * kSplitNct;
            if (u < rest) {
              float f[E];
              D::unpack(v[k][i], f);
#pragma unroll
              for (int e = 0; e < E; ++e) f[e] = __fmul_rn(exp_diff(f[e], ms), inv);
              st_stream16(yseg + (int64_t(k) * kPieceUnits + u) * 16, D::pack(f));
            }
          }
        }
      }
      if (c == 0 && tid == 0) {
        if (a.m_out) a.m_out[r] = row.m;
        if (a.d_out) a.d_out[r] = row.d;
        if (a.lse_out) a.lse_out[r] = lse_of(row);
      }
    }
    if (timed_out && lane == 0) atomicOr(a.status, kStatusTimeout);
  }
  __syncwarp();
  cluster_sync_all();  // no CTA leaves while a peer may still write into its shared memory
}

using SplitKernel = void (*)(SplitArgs);

SplitKernel split_kernel(int dtype) { return dtype == 0 ? k_splitrow<F32> : k_splitrow<BF16>; }

struct SplitPlan {
  bool ok = false;
  int cluster = 0;
  int clusters = 0;
  int slots = 0;
  size_t smem = 0;
};

std::mutex g_plan_mutex;
SplitPlan g_plan[64][2];
bool g_plan_ready[64][2];

// Cluster size and count giving the most resident CTAs (one per SM), and the ring size.
SplitPlan plan_for(int dtype, const DeviceInfo& dev) {
  std::lock_guard<std::mutex> lock(g_plan_mutex);
  if (dev.device >= 0 && dev.device < 64 && g_plan_ready[dev.device][dtype]) return g_plan[dev.device][dtype];
  SplitPlan best;
  if (dev.cluster_launch) {
    int slots = int((size_t(dev.max_smem_per_block_optin) - split_tail_bytes(16)) / kPieceBytes);
    if (slots > 16) slots = 16;
    const size_t smem = size_t(slots) * kPieceBytes + split_tail_bytes(slots);
    SplitKernel fn = split_kernel(dtype);
    if (slots >= 4 &&
        cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) == cudaSuccess) {
      for (int cs : {8, 4, 2}) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3((kSplitNcw + 1) * 32);
        cfg.dynamicSmemBytes = smem;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, (const void*)fn, &cfg) != cudaSuccess) {
          cudaGetLastError();
          continue;
        }
        if (n * cs > best.clusters * best.cluster) {
          best.ok = n > 0;
          best.cluster = cs;
          best.clusters = n;
          best.slots = slots;
          best.smem = smem;
        }
      }
    } else {
      cudaGetLastError();
    }
  }
  if (dev.device >= 0 && dev.device < 64) {
    g_plan[dev.device][dtype] = best;
    g_plan_ready[dev.device][dtype] = true;
  }
  return best;
}

}  // namespace

bool splitrow_fits(const RowProblem& p, const DeviceInfo& dev) {
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  if (row_bytes % 16 != 0) return false;
  const SplitPlan plan = plan_for(p.dtype, dev);
  if (!plan.ok) return false;
  const int64_t G = int64_t(plan.cluster) * plan.clusters;
  const int64_t units = row_bytes / 16;
  if (units < G * 64) return false;  // rows this short belong to the one-read kernels
  const int64_t seg = (units + G - 1) / G;
  return (seg + kPieceUnits - 1) / kPieceUnits <= (p.dtype == 0 ? max_pieces<F32>() : max_pieces<BF16>());
}

cudaError_t launch_splitrow(const RowProblem& p, const DeviceInfo& dev) {
  const SplitPlan plan = plan_for(p.dtype, dev);
  if (!plan.ok) return cudaErrorInvalidConfiguration;
  SplitKernel fn = split_kernel(p.dtype);
  cudaError_t err =
      cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(plan.smem));
  if (err != cudaSuccess) return err;
  const int G = plan.cluster * plan.clusters;
  // Scratch: one publication counter and the published cluster states, stream-ordered.
  const size_t state_bytes = size_t(p.M) * plan.clusters * 2 * sizeof(float);
  void* scratch = nullptr;
  if ((err = cudaMallocAsync(&scratch, 256 + state_bytes, p.stream)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(scratch, 0, 256, p.stream)) != cudaSuccess) {
    cudaFreeAsync(scratch, p.stream);
    return err;
  }
  SplitArgs a;
  a.x = static_cast<const unsigned char*>(p.x);
  a.y = static_cast<unsigned char*>(p.y);
  a.m_out = p.m_out;
  a.d_out = p.d_out;
  a.lse_out = p.lse_out;
  a.M = p.M;
  a.row_bytes = p.N * elem_bytes(p.dtype);
  a.units = a.row_bytes / 16;
  a.slots = plan.slots;
  a.counter = static_cast<unsigned*>(scratch);
  a.gstate = reinterpret_cast<float*>(static_cast<unsigned char*>(scratch) + 256);
  a.status = dev.status;
  a.local_wait_ns = local_wait_limit_ns();
  a.exchange_wait_ns = exchange_wait_limit_ns();
  a.fault = debug_fault();

  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(G);
  cfg.blockDim = dim3((kSplitNcw + 1) * 32);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = p.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, fn, a);
  cudaError_t ferr = cudaFreeAsync(scratch, p.stream);
  return err != cudaSuccess ? err : ferr;
}

}  // namespace rwo
