// kernel_splitrow.cu -- split-row softmax: few, very long rows spread over the whole GPU.
//
// "5.2 CUDA Online Softmax 实现优化" §7.1 names the case (small M, huge N: split one row over
// several blocks and merge their partial results); the merge is the (m, d) merge of §4.1, which
// is associative, so any partition of a row can be folded separately and combined.
//
// Layout: the grid is G persistent CTAs (one per SM), grouped in thread-block clusters of CS.
// Every row is cut into G contiguous segments of 16-byte units (pairs of CTAs split their share
// 48 : 52, see below); CTA c owns segment c of every row.  One producer lane streams the segments through a ring of shared-memory
// slots in 56 KB pieces with bulk copies (cp.async.bulk + mbarrier), each row's segment twice:
//
//   P1 -- the fold pass: loads marked L2::evict_last, so the lines stay in L2;
//   P2 -- the normalisation pass, issued once the row's exchange has completed: loads marked
//         evict_first, served from L2 (measured: DRAM reads stay at one read of x for 16 MiB rows).
//
// The producer picks each next piece: a P2 piece of the oldest row whose exchange is done, else a
// P1 piece of a row at most kL2Lag rows ahead of the oldest row still waiting for its P2, else the
// next P2 piece of that row before its exchange is done (its data does not depend on the
// exchange; only its arithmetic does).  Each slot carries a tag (row, piece, pass); the consumers
// follow the ring in order and wait for a row's state only at a P2 piece whose row's exchange is
// still running -- every P1 piece the exchange needs precedes it in the ring -- so HBM reads keep
// flowing while rows wait for their exchange and the first P2 pieces are already on chip when it
// completes.  Nothing
// of a row is held on chip, so the row length is not bounded by registers or shared memory (a row
// larger than L2 is still correct; its P2 then also reads HBM).
//
// Per row r, in every CTA:
//   1. P1 pieces: the thread's (m, d) state, folded a piece at a time (its values' maximum first,
//      one exponential per element, one rescale of the running sum per piece);
//   2. after the last P1 piece: warp butterfly merge, then cross-warp merge through shared memory
//      -> CTA state;
//   3. cluster merge over distributed shared memory: each CTA pushes its state into rank 0's
//      shared memory with st.async, which completes on rank 0's mbarrier as transaction bytes;
//      rank 0's producer lane, which polls that barrier while it waits, merges the CS states in
//      rank order and publishes the cluster state with one 64-bit release store into a
//      per-(row, cluster) slot;
//   4. the exchange warp (it issues no other global stores) polls the row's slots (acquire,
//      bounded by %globaltimer), merges all cluster states in a fixed order -- identical in
//      every CTA, so every CTA normalises with bitwise the same (m, d) -- and hands the row
//      state to the producer (and through the ring to the consumers) with an mbarrier;
//   5. P2 pieces: y = e^(x - m) / d, 16-byte stores.
// All clusters must be resident at once; the host launches at most the number of clusters the
// occupancy query reports.  Every wait is bounded; a wait that runs out records
// SOFTMAX_ERR_TIMEOUT in the status word, skips the remaining exchange waits, and the kernel
// still terminates.
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

// Warp roles: 14 consumer warps, 1 exchange warp, 1 producer warp = 16 warps (measured: faster
// than 30 consumer warps).  The exchange warp issues no global stores of its own, so its
// release operations never wait behind the row's output stores.
constexpr int kSplitNcw = 14;                                    // consumer warps
constexpr int kSplitNct = kSplitNcw * 32;                        // consumer threads
constexpr int kExchangeWarp = kSplitNcw;
constexpr int kProducerWarp = kSplitNcw + 1;
constexpr int kSplitThreads = (kSplitNcw + 2) * 32;
constexpr int kUnitsPerPiecePerThread = 8;  // measured: 56 KB pieces (4 slots) 200 us, 28 KB 210 us on 32 x 4 Mi fp32
constexpr int kPieceUnits = kSplitNct * kUnitsPerPiecePerThread;  // 3584 units
constexpr int kPieceBytes = kPieceUnits * 16;                    // 56 KB
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
                            // all ones (kUnpublished) until published -- set before launch
  unsigned* status;
  uint64_t local_wait_ns;
  uint64_t exchange_wait_ns;
  int fault;  // test hook: cluster 0 never publishes
};

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

// The publication slots read all ones until a state is written.  A published word is never all
// ones: a NaN d (a row holding NaN or +inf) is written as the canonical quiet NaN 0x7fffffff, so
// a row's NaN propagates into that row's outputs instead of looking unpublished.
constexpr unsigned long long kUnpublished = ~0ull;
__device__ __forceinline__ unsigned long long pack_state(State s) {
  const uint32_t d = s.d == s.d ? __float_as_uint(s.d) : 0x7fffffffu;
  return (static_cast<unsigned long long>(d) << 32) | __float_as_uint(s.m);
}

__device__ __forceinline__ State unpack_state(unsigned long long v) {
  return State{__uint_as_float(uint32_t(v)), __uint_as_float(uint32_t(v >> 32))};
}

// Online fold of one staged piece at piece granularity: the thread's values of the piece are
// loaded, their maximum taken first (packed for bf16), then one exponential per element with the
// packed f32x2 arithmetic, and one rescale of the running sum per piece.
template <class D, int UPT>
__device__ __forceinline__ State fold_piece(State st, uint32_t slot, int64_t rest, int tid) {
  constexpr int E = D::kVec;
  uint4 q[UPT];
#pragma unroll
  for (int i = 0; i < UPT; ++i) {
    const int u = tid + i * kSplitNct;
    q[i] = u < rest ? lds16(slot + uint32_t(u) * 16u)
                    : make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
  }
  const float m_new = fmaxf(st.m, D::vmax_all(q));
  const float ms = safe_max(m_new);
  float2 acc = make_float2(0.f, 0.f);
  float sum;
  if (exp_shift_ok(ms)) {
    const ExpShift sh = exp_shift(ms);
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
      float2 f[E / 2];
      D::unpack2(q[i], f);
#pragma unroll
      for (int e = 0; e < E / 2; ++e) acc = __fadd2_rn(acc, exp_shifted2(f[e], sh));
    }
    sum = __fmul_rn(__fadd_rn(acc.x, acc.y), sh.unscale);
  } else {
    const float2 nms = make_float2(-ms, -ms);
#pragma unroll
    for (int i = 0; i < UPT; ++i) {
      float2 f[E / 2];
      D::unpack2(q[i], f);
#pragma unroll
      for (int e = 0; e < E / 2; ++e) acc = __fadd2_rn(acc, exp_diff2(f[e], nms));
    }
    sum = __fadd_rn(acc.x, acc.y);
  }
  st.d = __fadd_rn(__fmul_rn(st.d, exp_diff(st.m, ms)), sum);
  st.m = m_new;
  return st;
}

__device__ __forceinline__ void cluster_sync_all() {
  // Non-aligned form: the producer warp's lanes reach it from different paths.
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

constexpr int kEvenSkewPermille = 40;  // the even CTA of a pair takes (1000 - 40) / 2000 of the pair's units
constexpr int kL2Lag = 2;    // P1 may run this many rows ahead of the oldest pending P2
constexpr int kRowBufs = 4;  // per-row buffers (states, barriers) in flight: kL2Lag + 2 <= 4
static_assert(kL2Lag + 2 <= kRowBufs, "row buffers must cover the rows in flight");

// Shared memory after the slots: full[S], freed[S], tag[S], cbar[4], cta_ready[4], row_ready[4],
// cstate[4][kMaxCluster], wstate[2][kSplitNcw], rowst[4].
size_t split_tail_bytes(int slots) {
  return size_t(slots) * 3 * sizeof(uint64_t) + 3 * kRowBufs * sizeof(uint64_t) +
         size_t(kRowBufs) * kMaxCluster * sizeof(State) + 2 * kSplitNcw * sizeof(State) + kRowBufs * sizeof(State);
}

template <class D>
__global__ void __launch_bounds__(kSplitThreads, 1) k_splitrow(SplitArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int E = D::kVec;
  constexpr int U = kUnitsPerPiecePerThread;
  constexpr int RB = kRowBufs;
  const int NS = a.slots;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(NS) * kPieceBytes);
  uint64_t* freed = full + NS;
  uint64_t* tag = freed + NS;            // [NS] (row << 32) | (piece << 1) | second
  uint64_t* cbar = tag + NS;             // [RB] cluster merge (rank 0)
  uint64_t* cta_ready = cbar + RB;       // [RB] consumers -> exchange warp
  uint64_t* row_ready = cta_ready + RB;  // [RB] exchange warp -> producer
  State* cstate = reinterpret_cast<State*>(row_ready + RB);  // [RB][kMaxCluster]
  State* wstate = cstate + RB * kMaxCluster;                 // [2][kSplitNcw]
  State* rowst = wstate + 2 * kSplitNcw;                     // [RB]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = cluster_nctarank();
  const uint32_t cid = cluster_id_x();
  const uint32_t ncl = cluster_count_x();

  const int64_t G = gridDim.x, c = blockIdx.x;
  // Segments: the row in G / 2 balanced pair shares, each split 48 : 52 between the even and the
  // odd CTA of the pair.  Measured (per-piece traces, 32 x 4 Mi fp32): with equal segments the
  // even CTA of each pair finished every row's P1 ~1.3 us after the odd one (a per-SM-pair
  // asymmetry), and each row's exchange waits for the slowest CTA; 4% fewer units for the even
  // CTA took 187.4 -> 185.5 us.  An odd G falls back to equal segments.
  int64_t seg_units, seg_start;
  if ((G & 1) == 0) {
    const int64_t P = G / 2, p = c / 2;
    const int64_t pbase = a.units / P, prem = a.units % P;
    const int64_t pu = pbase + (p < prem ? 1 : 0);          // >= 128 units (the host checks G * 64)
    const int64_t ps = p * pbase + (p < prem ? p : prem);
    const int64_t eu = pu * (1000 - kEvenSkewPermille) / 2000;
    seg_start = (c & 1) ? ps + eu : ps;
    seg_units = (c & 1) ? pu - eu : eu;
  } else {
    const int64_t base = a.units / G, rem = a.units % G;
    seg_units = base + (c < rem ? 1 : 0);
    seg_start = c * base + (c < rem ? c : rem);
  }
  const int64_t K = (seg_units + kPieceUnits - 1) / kPieceUnits;  // >= 1 (the host checks)
  const int64_t total = 2 * a.M * K;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&freed[s]), kSplitNcw);
    }
    for (int i = 0; i < RB; ++i) {
      mbar_init(smem_addr(&cbar[i]), 1);
      mbar_init(smem_addr(&cta_ready[i]), 1);
      mbar_init(smem_addr(&row_ready[i]), 1);
    }
    fence_mbar_init();
    if (crank == 0)
      for (int i = 0; i < RB && i < a.M; ++i) mbar_arrive_expect_tx(smem_addr(&cbar[i]), csize * 8u);
  }
  __syncthreads();
  cluster_sync_all();

  bool timed_out = false;
  if (warp == kProducerWarp) {
    if (lane == 0) {
      int64_t pubd = 0;
      auto service = [&]() {
        if (crank != 0) return;
        while (pubd < a.M && mbar_test(smem_addr(&cbar[pubd % RB]), uint32_t((pubd / RB) & 1)) &&
               mbar_test_cluster(smem_addr(&cbar[pubd % RB]), uint32_t((pubd / RB) & 1))) {
          State cs = empty_state();
          for (uint32_t i = 0; i < csize; ++i) cs = merge(cs, cstate[(pubd % RB) * kMaxCluster + i]);
          if (!(a.fault && cid == 0)) st_release_u64(a.pub + pubd * ncl + cid, pack_state(cs));
          if (pubd + RB < a.M) mbar_arrive_expect_tx(smem_addr(&cbar[pubd % RB]), csize * 8u);
          ++pubd;
        }
      };
      const uint64_t keep = policy_evict_last(), drop = policy_evict_first();
      int64_t r1 = 0, k1 = 0;  // next P1 piece
      int64_t r2 = 0, k2 = 0;  // next P2 piece
      bool ready2 = false;     // row r2's exchange is done
      int ps = 0;              // ring slot of piece n, and the parity of its lap (kept
      uint32_t pph = 0;        // incrementally: a 64-bit division per piece costs ~0.1 us)
      for (int64_t n = 0; n < total; ++n) {
        // choose the next piece: a P2 piece of a row whose exchange is done, else a P1 piece within
        // the lag, else the next P2 piece anyway -- its data does not depend on the exchange, so it
        // is loaded while the exchange finishes, and the consumers wait for the row's state
        if (!ready2) ready2 = mbar_test(smem_addr(&row_ready[r2 % RB]), uint32_t((r2 / RB) & 1));
        const bool second = ready2 || !(r1 < a.M && r1 <= r2 + kL2Lag);
        const int s = ps;
        if (n >= NS) {
          const uint32_t bar = smem_addr(&freed[s]);
          const uint32_t par = pph ^ 1u;  // the previous lap's release of this slot
          const uint64_t t1 = global_timer_ns();
          while (!mbar_test(bar, par)) {
            service();
            if (global_timer_ns() - t1 > a.local_wait_ns) {
              timed_out = true;
              break;
            }
          }
        }
        const int64_t r = second ? r2 : r1;
        const int64_t k = second ? k2 : k1;
        tag[s] = (uint64_t(r) << 32) | (uint64_t(k) << 1) | (second ? 1u : 0u);
        const int64_t rest = seg_units - k * kPieceUnits;
        const uint32_t bytes = uint32_t(rest < kPieceUnits ? rest : kPieceUnits) * 16u;
        const uint32_t bar = smem_addr(&full[s]);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(smem_addr(smem + size_t(s) * kPieceBytes), a.x + r * a.row_bytes + (seg_start + k * kPieceUnits) * 16,
                 bytes, bar, second ? drop : keep);
        if (second) {
          if (++k2 == K) {
            k2 = 0;
            ++r2;
            ready2 = false;
          }
        } else if (++k1 == K) {
          k1 = 0;
          ++r1;
        }
        if (++ps == NS) {
          ps = 0;
          pph ^= 1u;
        }
        service();
      }
      const uint64_t t0 = global_timer_ns();
      while (crank == 0 && pubd < a.M) {
        service();
        if (global_timer_ns() - t0 > a.local_wait_ns) {
          timed_out = true;
          break;
        }
      }
      for (int64_t n = total > NS ? total - NS : 0; n < total; ++n)  // once per launch
        if (!mbar_wait(smem_addr(&full[n % NS]), uint32_t((n / NS) & 1), a.local_wait_ns)) timed_out = true;
    }
  } else if (warp == kExchangeWarp) {
    bool abort = false;
    for (int64_t r = 0; r < a.M; ++r) {
      // every exit from this loop is taken by the whole warp: lane 0 alone reads the clock and
      // decides when the wait has run out (lanes that read the clock themselves could disagree at
      // the limit, and a lane that left would never reach the next full-warp collective)
      const uint64_t t0 = __shfl_sync(0xffffffffu, global_timer_ns(), 0);
      State g;
      while (true) {
        __syncwarp();
        bool ready = true;
        State gg = empty_state();
        if (!abort) {
          for (uint32_t i = lane; i < ncl; i += 32) {
            const unsigned long long v = ld_acquire_u64(a.pub + r * ncl + i);
            if (v == kUnpublished) ready = false;
            else gg = merge(gg, unpack_state(v));
          }
        }
        if (__all_sync(0xffffffffu, ready)) {
          g = warp_merge(gg);  // the same states in the same order in every CTA
          break;
        }
        const int expired = __shfl_sync(0xffffffffu, global_timer_ns() - t0 > a.exchange_wait_ns ? 1 : 0, 0);
        if (expired) {
          abort = true;
          timed_out = true;
          g = warp_merge(gg);
          break;
        }
        __nanosleep(20);
      }
      if (lane == 0) {
        // row r's buffer is free once this CTA handed over row r's state (it does so only after
        // the producer has issued every P2 piece of row r - RB + kL2Lag + 1 or later)
        if (!mbar_wait(smem_addr(&cta_ready[r % RB]), uint32_t((r / RB) & 1), a.local_wait_ns)) timed_out = true;
        rowst[r % RB] = g;
        mbar_arrive(smem_addr(&row_ready[r % RB]));
      }
    }
  } else {
    // ---------------- consumers: follow the ring ----------------
    State st = empty_state();  // fold of the P1 row in progress
    int cs = 0;                // ring slot of piece n and its lap parity
    uint32_t cph = 0;
    for (int64_t n = 0; n < total; ++n) {
      const int s = cs;
      const uint32_t par = cph;
      if (++cs == NS) {
        cs = 0;
        cph ^= 1u;
      }
      if (!mbar_wait(smem_addr(&full[s]), par, a.local_wait_ns)) timed_out = true;
      const uint64_t tg = tag[s];
      const int64_t r = int64_t(tg >> 32);
      const int64_t k = int64_t((tg & 0xffffffffu) >> 1);
      const uint32_t slot = smem_addr(smem + size_t(s) * kPieceBytes);
      const int64_t rest = seg_units - k * kPieceUnits;
      if (!(tg & 1u)) {
        // P1: fold the piece; after the row's last piece, the CTA state to the cluster
        st = fold_piece<D, kUnitsPerPiecePerThread>(st, slot, rest, tid);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&freed[s]));
        if (k == K - 1) {
          const State cs = group_merge(st, wstate + (r & 1) * kSplitNcw, kSplitNcw, warp, lane,
                                       [] { named_barrier_sync(1, kSplitNct); });
          if (tid == 0) {
            st_async_cluster_f32x2(map_to_rank(smem_addr(&cstate[(r % RB) * kMaxCluster + crank]), 0), cs.m, cs.d,
                                   map_to_rank(smem_addr(&cbar[r % RB]), 0));
            mbar_arrive(smem_addr(&cta_ready[r % RB]));
          }
          st = empty_state();
        }
      } else {
        // P2: normalise the re-read piece with the row's state and store y
        // the row's state (the piece may have been loaded before the row's exchange completed)
        if (!mbar_wait(smem_addr(&row_ready[r % RB]), uint32_t((r / RB) & 1), a.local_wait_ns)) timed_out = true;
        const State row = rowst[r % RB];
        const float ms = safe_max(row.m);
        const float inv = safe_inv(row.d);
        const float2 nms = make_float2(-ms, -ms), inv2 = make_float2(inv, inv);
        uint4 q[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
          const int u = tid + i * kSplitNct;
          if (u < rest) q[i] = lds16(slot + uint32_t(u) * 16u);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&freed[s]));
        unsigned char* yseg = a.y + r * a.row_bytes + (seg_start + k * kPieceUnits) * 16;
#pragma unroll
        for (int i = 0; i < U; ++i) {
          const int u = tid + i * kSplitNct;
          if (u < rest) {
            float2 f[E / 2];
            D::unpack2(q[i], f);
#pragma unroll
            for (int e = 0; e < E / 2; ++e) f[e] = __fmul2_rn(exp_diff2(f[e], nms), inv2);
            st_stream16(yseg + int64_t(u) * 16, D::pack2(f));
          }
        }
        if (k == 0 && c == 0 && tid == 0) {
          if (a.m_out) a.m_out[r] = row.m;
          if (a.d_out) a.d_out[r] = row.d;
          if (a.lse_out) a.lse_out[r] = lse_of(row);
        }
      }
    }
  }
  if (timed_out) atomicOr(a.status, kStatusTimeout);
  __syncwarp();
  cluster_sync_all();
}

using SplitKernel = void (*)(SplitArgs);

SplitKernel split_kernel(int dtype) {
  return dtype == 0 ? k_splitrow<F32> : dtype == 1 ? k_splitrow<BF16> : k_splitrow<F16>;
}

struct SplitPlan {
  bool ok = false;
  int cluster = 0;
  int clusters = 0;
  int slots = 0;
  size_t smem = 0;
};

std::mutex g_plan_mutex;
SplitPlan g_plan[64][3];
bool g_plan_ready[64][3];

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
  return true;  // nothing of a row is held on chip: any length
}

size_t splitrow_slots(const RowProblem& p, const DeviceInfo& dev) {
  const SplitPlan plan = plan_for(p.dtype, dev);
  return plan.ok ? size_t(p.M) * plan.clusters : 0;
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
