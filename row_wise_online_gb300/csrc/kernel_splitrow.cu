// kernel_splitrow.cu -- split-row softmax: few, very long rows spread over the whole GPU.
//
// "5.2 CUDA Online Softmax 实现优化" §7.1 names the case (small M, huge N: split one row over
// several blocks and merge their partial results); the merge is the (m, d) merge of §4.1, which
// is associative, so any partition of a row can be folded separately and combined.
//
// Layout: the grid is G persistent CTAs (one per SM), grouped in thread-block clusters of CS.
// Every row is cut into G contiguous segments of 16-byte units, balanced to one unit; CTA c owns
// segment c of every row.  One producer lane streams the segments of consecutive rows, in 14 KB
// pieces, through a ring of shared-memory slots with bulk copies (cp.async.bulk + mbarrier).
// Consumers keep row r's segment in registers (up to 8 pieces, 2 vectors per thread per piece)
// while its exchange is in flight, fold row r + 1 straight from its staged slots, and then,
// piece by piece, normalise row r from registers and gather row r + 1 into the registers just
// freed, handing each slot back to the producer.  x is read once; y is written once, straight
// from registers.
//
// Per row r, in every CTA:
//   1. the thread's (m, d) state: online fold over its units (one rescale per 16-byte unit, one
//      exponential per element);
//   2. warp butterfly merge, then cross-warp merge through shared memory -> CTA state;
//   3. cluster merge over distributed shared memory: each CTA pushes its state into rank 0's
//      shared memory with st.async, which completes on rank 0's mbarrier as transaction bytes
//      (no fence, so it never waits behind the row's output stores); rank 0's producer lane,
//      which polls that barrier while it waits for free slots, merges the CS states in rank
//      order and publishes the cluster state with one 64-bit release store into a
//      per-(row, cluster) slot;
//   4. the exchange warp (it issues no other global stores) polls the row's slots (acquire,
//      bounded by %globaltimer), merges all cluster states in a fixed order -- identical in
//      every CTA, so every CTA normalises with bitwise the same (m, d) -- and hands the row
//      state to the consumers through an mbarrier;
//   5. y = e^(x - m) / d from registers, 16-byte stores.
// Row r + 1 is published before row r is awaited, so the exchange of one row overlaps the work
// of the next.
// All clusters must be resident at once; the host launches at most the number of clusters the
// occupancy query reports.  Every wait is bounded; a wait that runs out records
// SOFTMAX_ERR_TIMEOUT in the status word, skips the remaining exchange waits, and the kernel
// still terminates.
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

// Warp roles: 14 consumer warps, 1 exchange warp, 1 producer warp = 16 warps, 4 per SM
// sub-partition, so each thread may use up to 128 registers (17 warps would cap it at 96 and
// spill the row).  The exchange warp issues no global stores of its own, so its release
// operations never wait behind the row's output stores.
constexpr int kSplitNcw = 14;                                    // consumer warps
constexpr int kSplitNct = kSplitNcw * 32;                        // consumer threads
constexpr int kExchangeWarp = kSplitNcw;
constexpr int kProducerWarp = kSplitNcw + 1;
constexpr int kSplitThreads = (kSplitNcw + 2) * 32;
constexpr int kUnitsPerPiecePerThread = 2;
constexpr int kPieceUnits = kSplitNct * kUnitsPerPiecePerThread;  // 896 units
constexpr int kPieceBytes = kPieceUnits * 16;                    // 14 KB
// Register capacity per CTA and row: 8 pieces (112 KB) for fp32; 6 for bf16, whose unpacking
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
  unsigned long long* pub;  // [M][clusters] published cluster states (m, d) as one 64-bit word;
                            // all-ones (NaN) until published -- set before launch
  unsigned* status;
  uint64_t local_wait_ns;
  uint64_t exchange_wait_ns;
  int fault;  // test hook: cluster 0 never publishes
};

// Shared memory after the slots: full[S], freed[S], cbar[2], cta_ready[2], row_ready[2],
// cstate[2][kMaxCluster], wstate[2][kSplitNcw], rowst[2].
size_t split_tail_bytes(int slots) {
  return size_t(slots) * 2 * sizeof(uint64_t) + 6 * sizeof(uint64_t) + 2 * kMaxCluster * sizeof(State) +
         2 * kSplitNcw * sizeof(State) + 2 * sizeof(State);
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Asynchronous store of (a, b) into shared memory of a CTA of this cluster; completion is
// counted as 8 transaction bytes on the mbarrier `mbar` (also in that CTA).  No fence: it does
// not wait for this thread's earlier global stores.
__device__ __forceinline__ void st_async_cluster_f32x2(uint32_t addr, float a, float b, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "f"(a), "f"(b), "r"(mbar)
               : "memory");
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long pack_state(State s) {
  return (static_cast<unsigned long long>(__float_as_uint(s.d)) << 32) | __float_as_uint(s.m);
}

__device__ __forceinline__ State unpack_state(unsigned long long v) {
  return State{__uint_as_float(uint32_t(v)), __uint_as_float(uint32_t(v >> 32))};
}

// Online fold of the units this thread owns in one staged piece: per 16-byte unit, one
// rescale of the running sum and one exponential per element (the recurrence, unit-wise).
template <class D>
__device__ __forceinline__ State fold_piece_smem(State st, uint32_t slot, int64_t rest, int tid) {
  constexpr int E = D::kVec;
#pragma unroll
  for (int i = 0; i < kUnitsPerPiecePerThread; ++i) {
    const int u = tid + i * kSplitNct;
    if (u < rest) {
      const uint4 q = lds16(slot + uint32_t(u) * 16u);
      float f[E];
      D::unpack(q, f);
      const float m_new = fmaxf(st.m, D::vmax(q));
      const float ms = safe_max(m_new);
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc += exp_diff(f[e], ms);
      st.d = __fadd_rn(__fmul_rn(st.d, exp_diff(st.m, ms)), acc);
      st.m = m_new;
    }
  }
  return st;
}

__device__ __forceinline__ void cluster_sync_all() {
  // Non-aligned form: the producer warp's lanes reach it from different paths.
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

template <class D>
__global__ void __launch_bounds__(kSplitThreads, 1) k_splitrow(SplitArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int E = D::kVec;
  constexpr int U = kUnitsPerPiecePerThread;
  constexpr int KMAX = max_pieces<D>();
  const int NS = a.slots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(NS) * kPieceBytes);
  uint64_t* freed = full + NS;
  uint64_t* cbar = freed + NS;          // [2] cluster merge (used in rank 0), count = cluster size
  uint64_t* cta_ready = cbar + 2;       // [2] consumers -> exchange warp: row's CTA state sent
  uint64_t* row_ready = cta_ready + 2;  // [2] exchange warp -> consumers: row state is in rowst
  State* cstate = reinterpret_cast<State*>(row_ready + 2);  // [2][kMaxCluster], written into rank 0
  State* wstate = cstate + 2 * kMaxCluster;                 // [2][kSplitNcw]
  State* rowst = wstate + 2 * kSplitNcw;                    // [2]

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
  const int K = int((seg_units + kPieceUnits - 1) / kPieceUnits);  // <= KMAX, 2K <= NS (the host checks)

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&freed[s]), kSplitNcw);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&cbar[i]), 1);
      mbar_init(smem_addr(&cta_ready[i]), 1);
      mbar_init(smem_addr(&row_ready[i]), 1);
    }
    fence_mbar_init();
    // rank 0 expects csize states of 8 bytes for each of rows 0 and 1 (re-armed per row)
    if (crank == 0)
      for (int i = 0; i < 2 && i < a.M; ++i) mbar_arrive_expect_tx(smem_addr(&cbar[i]), csize * 8u);
  }
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before any remote arrive

  bool timed_out = false;
  if (warp == kProducerWarp) {
    // ---------------- producer: stream pieces of consecutive rows through the ring ----------------
    // In rank 0 the same lane also merges and publishes the cluster's state of each row as soon
    // as all of the cluster's states have landed: it polls that barrier while it waits for free
    // slots, and it issues no generic global stores, so its release store is not held up.
    if (lane == 0) {
      int64_t pubd = 0;
      auto service = [&]() {
        if (crank != 0) return;
        while (pubd < a.M && mbar_test_cluster(smem_addr(&cbar[pubd & 1]), uint32_t((pubd >> 1) & 1))) {
          State cs = empty_state();
          for (uint32_t i = 0; i < csize; ++i) cs = merge(cs, cstate[(pubd & 1) * kMaxCluster + i]);
          if (!(a.fault && cid == 0)) st_release_u64(a.pub + pubd * ncl + cid, pack_state(cs));
          if (pubd + 2 < a.M) mbar_arrive_expect_tx(smem_addr(&cbar[pubd & 1]), csize * 8u);  // row pubd + 2
          ++pubd;
        }
      };
      const uint64_t pol = policy_evict_first();
      const int64_t total = K > 0 ? a.M * K : 0;
      for (int64_t p = 0; p < total; ++p) {
        const int s = int(p % NS);
        if (p >= NS) {
          const uint32_t bar = smem_addr(&freed[s]);
          const uint32_t par = uint32_t(((p / NS) - 1) & 1);
          const uint64_t t0 = global_timer_ns();
          while (!mbar_test(bar, par)) {
            service();
            if (global_timer_ns() - t0 > a.local_wait_ns) {
              timed_out = true;
              break;
            }
          }
        }
        const int64_t r = p / K;
        const int k = int(p % K);
        const int64_t rest = seg_units - int64_t(k) * kPieceUnits;
        const uint32_t bytes = uint32_t(rest < kPieceUnits ? rest : kPieceUnits) * 16u;
        const uint32_t bar = smem_addr(&full[s]);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(smem_addr(smem + size_t(s) * kPieceBytes),
                 a.x + r * a.row_bytes + (seg_start + int64_t(k) * kPieceUnits) * 16, bytes, bar, pol);
        service();
      }
      // rank 0: publish the remaining rows (bounded: a peer that timed out may never send)
      const uint64_t t0 = global_timer_ns();
      while (crank == 0 && pubd < a.M) {
        service();
        if (global_timer_ns() - t0 > a.local_wait_ns) {
          timed_out = true;
          break;
        }
      }
      // every load has landed before the CTA may exit (the consumers normally saw them all)
      for (int64_t p = total > NS ? total - NS : 0; p < total; ++p)
        if (!mbar_wait(smem_addr(&full[p % NS]), uint32_t((p / NS) & 1), a.local_wait_ns)) timed_out = true;
    }
  } else if (warp == kExchangeWarp) {
    // ---------------- exchange: wait across clusters ----------------
    // All lanes poll the published cluster states of the row being awaited (the consumers
    // push CTA states into rank 0 with st.async; rank 0's producer lane publishes).
    bool abort = false;
    for (int64_t r = 0; r < a.M; ++r) {
      const uint64_t t0 = global_timer_ns();
      State g;
      while (true) {
        __syncwarp();
        bool ready = true;
        State gg = empty_state();
        if (!abort) {
          for (uint32_t i = lane; i < ncl; i += 32) {
            const State cs = unpack_state(ld_acquire_u64(a.pub + r * ncl + i));
            if (cs.d != cs.d) ready = false;  // NaN: not published yet
            else gg = merge(gg, cs);
          }
        }
        if (__all_sync(0xffffffffu, ready)) {
          g = warp_merge(gg);  // every CTA merges the same states in the same order
          break;
        }
        if (global_timer_ns() - t0 > a.exchange_wait_ns) {
          abort = true;  // later rows do not wait again
          timed_out = true;
          g = warp_merge(gg);
          break;
        }
        __nanosleep(20);
      }
      if (lane == 0) {
        // Signal row r only once the consumers have handed over row r's state: they do that after
        // consuming row r - 2's signal, so one buffer never completes two phases ahead of its
        // waiters (this already holds when the exchange did not run out).
        if (!mbar_wait(smem_addr(&cta_ready[r & 1]), uint32_t((r >> 1) & 1), a.local_wait_ns)) timed_out = true;
        rowst[r & 1] = g;
        mbar_arrive(smem_addr(&row_ready[r & 1]));
      }
    }
  } else {
    // ---------------- consumers ----------------
    // Registers hold row r while it waits for its exchange; row r + 1 is folded straight from
    // its staged slots and handed to the exchange warp first, so exchanges overlap a row of work.
    uint4 v[KMAX][U];
    auto publish = [&](int64_t r, State st) {
      st = group_merge(st, wstate + (r & 1) * kSplitNcw, kSplitNcw, warp, lane,
                       [] { named_barrier_sync(1, kSplitNct); });
      if (tid == 0) {
        st_async_cluster_f32x2(map_to_rank(smem_addr(&cstate[(r & 1) * kMaxCluster + crank]), 0), st.m, st.d,
                               map_to_rank(smem_addr(&cbar[r & 1]), 0));
        mbar_arrive(smem_addr(&cta_ready[r & 1]));
      }
    };
    // prologue: row 0 into registers, then its state
    if (a.M > 0) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k) {
#pragma unroll
        for (int i = 0; i < U; ++i) v[k][i] = make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
        if (k < K) {
          const int s = k % NS;
          if (!mbar_wait(smem_addr(&full[s]), 0u, a.local_wait_ns)) timed_out = true;
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
      publish(0, State{mt, dt});
    }
    for (int64_t r = 0; r < a.M; ++r) {
      const bool more = r + 1 < a.M;
      // 1. fold row r + 1 from its slots and hand its state over
      if (more) {
        State st = empty_state();
        for (int k = 0; k < K; ++k) {
          const int64_t p = (r + 1) * K + k;
          const int s = int(p % NS);
          if (!mbar_wait(smem_addr(&full[s]), uint32_t((p / NS) & 1), a.local_wait_ns)) timed_out = true;
          st = fold_piece_smem<D>(st, smem_addr(smem + size_t(s) * kPieceBytes),
                                  seg_units - int64_t(k) * kPieceUnits, tid);
        }
        publish(r + 1, st);
      }
      // 2. row r's state
      if (!mbar_wait(smem_addr(&row_ready[r & 1]), uint32_t((r >> 1) & 1), a.local_wait_ns)) timed_out = true;
      const State row = rowst[r & 1];
      const float ms = safe_max(row.m);
      const float inv = safe_inv(row.d);
      // 3. piece by piece: normalise row r from registers and store, then gather row r + 1's
      //    piece into the registers just freed and hand its slot back
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
          if (more) {
            const int64_t p = (r + 1) * K + k;
            const int s = int(p % NS);
            const uint32_t slot = smem_addr(smem + size_t(s) * kPieceBytes);
#pragma unroll
            for (int i = 0; i < U; ++i) {
              const int u = tid + i * kSplitNct;
              if (u < rest) v[k][i] = lds16(slot + uint32_t(u) * 16u);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&freed[s]));
          }
        }
      }
      if (c == 0 && tid == 0) {
        if (a.m_out) a.m_out[r] = row.m;
        if (a.d_out) a.d_out[r] = row.d;
        if (a.lse_out) a.lse_out[r] = lse_of(row);
      }
    }
  }
  if (timed_out) atomicOr(a.status, kStatusTimeout);
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
        cfg.blockDim = dim3(kSplitThreads);
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
  const int64_t K = (seg + kPieceUnits - 1) / kPieceUnits;
  return K <= (p.dtype == 0 ? max_pieces<F32>() : max_pieces<BF16>()) && 2 * K <= plan.slots;
}

cudaError_t launch_splitrow(const RowProblem& p, const DeviceInfo& dev) {
  const SplitPlan plan = plan_for(p.dtype, dev);
  if (!plan.ok) return cudaErrorInvalidConfiguration;
  SplitKernel fn = split_kernel(p.dtype);
  cudaError_t err =
      cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(plan.smem));
  if (err != cudaSuccess) return err;
  const int G = plan.cluster * plan.clusters;
  // Scratch: one 64-bit publication slot per (row, cluster), stream-ordered, all-ones until published.
  const size_t pub_bytes = size_t(p.M) * plan.clusters * sizeof(unsigned long long);
  void* scratch = nullptr;
  if ((err = cudaMallocAsync(&scratch, pub_bytes, p.stream)) != cudaSuccess) return err;
  if ((err = cudaMemsetAsync(scratch, 0xFF, pub_bytes, p.stream)) != cudaSuccess) {
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
  a.pub = static_cast<unsigned long long*>(scratch);
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
  cfg.blockDim = dim3(kSplitThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = p.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, fn, a);
  cudaError_t ferr = cudaFreeAsync(scratch, p.stream);
  return err != cudaSuccess ? err : ferr;
}

cudaError_t launch_splitrow_scratch(const RowProblem& p, const DeviceInfo& dev, unsigned long long* pub,
                                    size_t pub_slots, bool* too_big) {
  *too_big = false;
  const SplitPlan plan = plan_for(p.dtype, dev);
  if (!plan.ok) return cudaErrorInvalidConfiguration;
  const size_t need = size_t(p.M) * plan.clusters;
  if (need > pub_slots) {
    *too_big = true;
    return cudaErrorInvalidValue;
  }
  SplitKernel fn = split_kernel(p.dtype);
  cudaError_t err =
      cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(plan.smem));
  if (err != cudaSuccess) return err;
  // The slots must read as "not published" (all ones) when the kernel starts.
  if ((err = cudaMemsetAsync(pub, 0xFF, need * sizeof(unsigned long long), p.stream)) != cudaSuccess) return err;
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
  a.pub = pub;
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
  cfg.gridDim = dim3(plan.cluster * plan.clusters);
  cfg.blockDim = dim3(kSplitThreads);
  cfg.dynamicSmemBytes = plan.smem;
  cfg.stream = p.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace rwo
