// kernel_splitrow_onchip.cu -- split-row softmax with each CTA's segment held on chip: one read.
//
// "5.2 CUDA Online Softmax 实现优化" §7.1 names the case (small M, huge N: several blocks share a
// row and merge their partial results); the merge is the (m, d) merge of §4.1, associative, so
// any partition of a row can be folded separately and combined.
//
// The grid is G persistent CTAs, one per SM, in thread-block clusters of CS.  Every row is cut
// into G contiguous segments of 16-byte units; CTA c owns segment c of every row.  The segment
// stays in shared memory from its load until its normalisation, so x is read from HBM once and
// the normalisation reads shared memory instead of L2 (the streaming split-row kernel reads each
// segment twice).  A 16 MiB row over 152 SMs is ~110 KB per CTA; NB row buffers of that size
// (NB = 2 for such rows, up to 8 for shorter ones) are resident, so the fold of the next rows and
// their loads overlap the exchange of a row's state.
//
// Roles (one CTA):
//   * producer lane: bulk copies (cp.async.bulk + mbarrier) of row r's segment, in pieces of
//     32 KB, into buffer r mod NB as soon as the consumers have normalised that buffer's previous
//     row piece by piece (each piece has its own full / freed barriers);
//   * consumer warps: for row r + NB - 1 then row r (a lag of NB - 1 rows): fold each piece of the
//     row's segment as it lands (thread max first, one exponential per element, one rescale per
//     piece), warp and cross-warp merges to the CTA state, pushed with st.async into rank 0's
//     shared memory, where it completes as transaction bytes on rank 0's per-row barrier; then,
//     once row r's state is known, y = e^(x - m) / d from the held segment, 16-byte stores, and
//     each piece freed for the producer;
//   * exchange warp: on rank 0, waits for the cluster's CS states (bounded), merges them in rank
//     order and publishes the cluster state with one 64-bit release store into a per-(row,
//     cluster) slot; on every CTA, polls the row's slots (acquire, bounded by %globaltimer),
//     merges all cluster states in a fixed order -- identical in every CTA, so every CTA
//     normalises with bitwise the same (m, d) -- and hands the row state to the consumers.
//
// Buffer reuse needs no extra synchronisation: a CTA's state for row r + NB is pushed only after
// every consumer of that CTA has finished normalising row r (the cross-warp merge's barrier lies
// between them), so the per-row barriers and state slots of buffer r mod NB are free again by the
// time row r + NB reaches them, and a barrier is never more than one phase ahead of its waiter.
// All clusters must be resident at once; the host launches at most the number of clusters the
// occupancy query reports.  Every wait is bounded; a wait that runs out records
// SOFTMAX_ERR_TIMEOUT in the status word, later exchange waits are skipped, and the kernel still
// terminates.
#include <mutex>

#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

constexpr int kOcNcw = 16;                         // consumer warps
constexpr int kOcNct = kOcNcw * 32;                // consumer threads
constexpr int kOcExchangeWarp = kOcNcw;
constexpr int kOcProducerWarp = kOcNcw + 1;
constexpr int kOcPublisherWarp = kOcNcw + 2;       // rank 0 of a cluster: merges and publishes
constexpr int kOcThreads = (kOcNcw + 3) * 32;
constexpr int kOcUpt = 4;                          // 16-byte units per consumer thread per piece
constexpr int kOcPieceUnits = kOcNct * kOcUpt;     // 2048 units
constexpr int kOcPieceBytes = kOcPieceUnits * 16;  // 32 KB
constexpr int kOcMaxBufs = 8;
constexpr int kOcMaxPieces = 8;
constexpr int kOcMaxCluster = 16;  // cluster states per row slot (clusters of up to 16 in local mode)
constexpr int kOcPrefetchRows = 1;  // L2 prefetch distance in rows (measured on 32 x 16 MiB fp32: 170 us; 2 rows 176, 3 rows 200, none 190)

struct OnchipArgs {
  const unsigned char* x;
  unsigned char* y;
  float* m_out;
  float* d_out;
  float* lse_out;
  int64_t M;
  int64_t units;      // 16-byte units per row
  int64_t row_bytes;
  int nb;             // shared-memory row buffers
  int rb;             // row-state slots (rows between their fold and their normalisation)
  int pieces;         // pieces per buffer (of the longest segment)
  uint32_t buf_bytes; // bytes per row buffer
  unsigned long long* pub;  // [M][clusters] published cluster states; all ones until published
  unsigned* status;
  uint64_t local_wait_ns;
  uint64_t exchange_wait_ns;
  int fault;  // test hook: cluster 0 never publishes
  int local;  // each cluster owns whole rows (cid, cid + clusters, ...): the state is merged over DSMEM only
};

constexpr unsigned long long kOcUnpublished = ~0ull;

// A published word is never all ones: a NaN d (a row holding NaN or +inf) is written as the
// canonical quiet NaN 0x7fffffff, so that row's NaN reaches its outputs instead of reading as
// "not yet published".
__device__ __forceinline__ unsigned long long oc_pack(State s) {
  const uint32_t d = s.d == s.d ? __float_as_uint(s.d) : 0x7fffffffu;
  return (static_cast<unsigned long long>(d) << 32) | __float_as_uint(s.m);
}

__device__ __forceinline__ State oc_unpack(unsigned long long v) {
  return State{__uint_as_float(uint32_t(v)), __uint_as_float(uint32_t(v >> 32))};
}

__device__ __forceinline__ void oc_st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long oc_ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// st.async of (a, b) into shared memory of a CTA of this cluster, completing as 8 transaction
// bytes on the mbarrier `mbar` of that CTA.
__device__ __forceinline__ void oc_st_async_f32x2(uint32_t addr, float a, float b, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
               "f"(a), "f"(b), "r"(mbar)
               : "memory");
}

// Bulk prefetch of global memory into L2 (no shared memory, no completion to wait for).
__device__ __forceinline__ void oc_prefetch_l2(const void* src, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes), "l"(policy)
               : "memory");
}

__device__ __forceinline__ uint32_t oc_cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void oc_cluster_sync_all() {
  // non-aligned form: the producer warp's lanes reach it from different paths
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Fold of one landed piece: the thread's units (u = tid + i * kOcNct), their maximum first, then
// one exponential per element with packed f32x2 arithmetic and one rescale of the running sum.
template <class D>
__device__ __forceinline__ State oc_fold_piece(State st, uint32_t piece, int rest, int tid) {
  constexpr int E = D::kVec;
  uint4 q[kOcUpt];
#pragma unroll
  for (int i = 0; i < kOcUpt; ++i) {
    const int u = tid + i * kOcNct;
    q[i] = u < rest ? lds16(piece + uint32_t(u) * 16u)
                    : make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
  }
  const float m_new = fmaxf(st.m, D::vmax_all(q));
  const float ms = safe_max(m_new);
  float2 acc = make_float2(0.f, 0.f);
  float sum;
  if (exp_shift_ok(ms)) {
    const ExpShift sh = exp_shift(ms);
#pragma unroll
    for (int i = 0; i < kOcUpt; ++i) {
      float2 f[E / 2];
      D::unpack2(q[i], f);
#pragma unroll
      for (int e = 0; e < E / 2; ++e) acc = __fadd2_rn(acc, exp_shifted2(f[e], sh));
    }
    sum = __fmul_rn(__fadd_rn(acc.x, acc.y), sh.unscale);
  } else {
    const float2 nms = make_float2(-ms, -ms);
#pragma unroll
    for (int i = 0; i < kOcUpt; ++i) {
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

// Position in a ring of n entries, kept incrementally (no 64-bit division per row): the entry of
// row r and how many times the ring wrapped before it (the mbarrier phase parity is lap & 1).
struct OcRing {
  int idx = 0;
  int64_t lap = 0;
  int n;
  __device__ explicit OcRing(int entries) : n(entries) {}
  __device__ void next() {
    if (++idx == n) {
      idx = 0;
      ++lap;
    }
  }
  __device__ uint32_t parity() const { return uint32_t(lap & 1); }
};

// Tensor memory when segments are parked there (HOLD): 2 row slots of 256 columns; warp w owns
// lanes 32 (w mod 4) .. + 31 and columns 64 (w / 4) .. + 63 of a slot, one lane per thread: thread
// t's unit i = 4 p + k (unit p * kOcPieceUnits + k * kOcNct + t of the segment) in columns 4 i .. 4 i + 3.
constexpr uint32_t kOcTmemCols = 512;
constexpr uint32_t kOcSlotCols = 256;
constexpr uint32_t kOcWarpCols = 64;
static_assert(kOcNcw / 4 * kOcWarpCols == kOcSlotCols, "a slot's columns cover the consumer warps");
static_assert(kOcMaxPieces * kOcUpt * 4 >= kOcWarpCols, "pieces per segment bounded by the columns");

__device__ __forceinline__ void oc_tmem_st16(uint32_t taddr, const uint4 (&q)[kOcUpt]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(q[0].x), "r"(q[0].y), "r"(q[0].z), "r"(q[0].w), "r"(q[1].x), "r"(q[1].y), "r"(q[1].z), "r"(q[1].w),
      "r"(q[2].x), "r"(q[2].y), "r"(q[2].z), "r"(q[2].w), "r"(q[3].x), "r"(q[3].y), "r"(q[3].z), "r"(q[3].w)
      : "memory");
}
__device__ __forceinline__ void oc_tmem_ld16(uint32_t taddr, uint4 (&q)[kOcUpt]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(q[0].x), "=r"(q[0].y), "=r"(q[0].z), "=r"(q[0].w), "=r"(q[1].x), "=r"(q[1].y), "=r"(q[1].z),
        "=r"(q[1].w), "=r"(q[2].x), "=r"(q[2].y), "=r"(q[2].z), "=r"(q[2].w), "=r"(q[3].x), "=r"(q[3].y),
        "=r"(q[3].z), "=r"(q[3].w)
      : "r"(taddr));
}
__device__ __forceinline__ void oc_tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void oc_tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void oc_tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void oc_tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared memory after the row buffers: full[NB][P], freed[NB][P], cbar[RB], row_ready[RB],
// cstate[RB][kOcMaxCluster], wstate[2][kOcNcw], rowst[RB], the tensor-memory address.
size_t onchip_tail_bytes(int nb, int rb, int pieces) {
  return size_t(nb) * pieces * 2 * sizeof(uint64_t) + size_t(rb) * 2 * sizeof(uint64_t) +
         size_t(rb) * kOcMaxCluster * sizeof(State) + 2 * kOcNcw * sizeof(State) + size_t(rb) * sizeof(State) + 16;
}

// HOLD: one or two shared-memory buffers (landing and fold), segments parked in tensor memory until
// their row state arrives; else NB shared-memory buffers, fold NB - 1 rows ahead of the normalisation.
// Split mode (local = 0): every row is shared by all G CTAs, cluster states exchanged through global
// memory.  Local mode: cluster k owns rows k, k + clusters, ... and its CS CTAs share each of them;
// rank 0 merges the CTA states and hands the row state to every CTA of the cluster over DSMEM.
template <class D, bool HOLD, bool LOG>
__global__ void __launch_bounds__(kOcThreads, 1) k_splitrow_onchip(OnchipArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int E = D::kVec;
  const int NB = a.nb, P = a.pieces, RB = a.rb;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(NB) * a.buf_bytes);  // [NB][P]
  uint64_t* freed = full + NB * P;                                                  // [NB][P]
  uint64_t* cbar = freed + NB * P;                                                  // [RB] (rank 0)
  uint64_t* row_ready = cbar + RB;                                                  // [RB]
  State* cstate = reinterpret_cast<State*>(row_ready + RB);                         // [RB][kOcMaxCluster]
  State* wstate = cstate + RB * kOcMaxCluster;                                      // [2][kOcNcw]
  State* rowst = wstate + 2 * kOcNcw;                                               // [RB]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rowst + RB);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t csize = oc_cluster_nctarank();
  const uint32_t cid = cluster_id_x();
  const uint32_t ncl = cluster_count_x();
  const bool local = a.local != 0;
  // the rows this CTA takes part in: M of them, the j-th is row_of(j)
  const int64_t M = local ? (a.M > int64_t(cid) ? (a.M - 1 - cid) / ncl + 1 : 0) : a.M;
  auto row_of = [&](int64_t j) { return local ? int64_t(cid) + j * int64_t(ncl) : j; };

  // this CTA's segment: units [seg_start, seg_start + seg_units) of every row (measured: giving the
  // even CTA of each SM pair 4% fewer units, as the streaming kernel does, changes nothing here)
  const int64_t G = local ? int64_t(csize) : int64_t(gridDim.x), c = local ? int64_t(crank) : int64_t(blockIdx.x);
  const int64_t base = a.units / G, rem = a.units % G;
  const int seg_units = int(base + (c < rem ? 1 : 0));
  const int64_t seg_start = c * base + (c < rem ? c : rem);
  const int pc = (seg_units + kOcPieceUnits - 1) / kOcPieceUnits;  // pieces of this CTA's segment, <= P

  if (tid == 0) {
    for (int i = 0; i < NB * P; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&freed[i]), kOcNcw);
    }
    for (int i = 0; i < RB; ++i) {
      mbar_init(smem_addr(&cbar[i]), 1);
      mbar_init(smem_addr(&row_ready[i]), 1);
    }
    fence_mbar_init();
    if (crank == 0)
      for (int i = 0; i < RB && i < M; ++i) mbar_arrive_expect_tx(smem_addr(&cbar[i]), csize * 8u);
  }
  if constexpr (HOLD) {
    if (warp == 0) {  // all 512 columns: one CTA per SM (its shared memory admits no second one)
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                   "n"(kOcTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    oc_tc_fence_before();
  }
  __syncthreads();
  if constexpr (HOLD) oc_tc_fence_after();
  oc_cluster_sync_all();

  bool timed_out = false;
  // after a wait of this thread has run out, its later waits on this CTA's own copies and threads
  // are cut short (the result is already void), so a broken launch ends in about one wait limit;
  // the producer's final drain keeps the full limit
  uint64_t lim = a.local_wait_ns;
  const uint32_t bufs = smem_addr(smem);
  if (warp == kOcProducerWarp) {
    if (lane == 0) {
      const uint64_t drop = policy_evict_first();  // x is read once
      const uint64_t keep = policy_evict_last();   // prefetched lines wait in L2 for their load
      // Row r + PD is prefetched into L2 when row r's loads are issued (rows NB .. NB + PD - 1
      // right after the first NB rows' loads, which go first so that the first fold starts
      // early): HBM reads run PD rows ahead of the buffers, so a buffer freed by the consumers
      // refills from L2 instead of waiting for HBM, and the reads of later rows fill the time
      // the first rows wait for their exchange.
      const int PD = kOcPrefetchRows;
      OcRing ring(NB);
      for (int64_t r = 0; r < M; ++r) {
        const int b = ring.idx;
        const int64_t lap = ring.lap;
        const unsigned char* src = a.x + row_of(r) * a.row_bytes + seg_start * 16;
        const bool pf = PD > 0 && lap > 0 && r + PD < M;  // rows NB .. NB + PD - 1: after the first loads
        if (r == NB)
          for (int64_t q = NB; q < NB + int64_t(PD) && q < M; ++q)
            for (int p = 0; p < pc; ++p) {
              const int rest = seg_units - p * kOcPieceUnits;
              oc_prefetch_l2(a.x + row_of(q) * a.row_bytes + seg_start * 16 + int64_t(p) * kOcPieceBytes,
                             uint32_t(rest < kOcPieceUnits ? rest : kOcPieceUnits) * 16u, keep);
            }
        for (int p = 0; p < pc; ++p) {
          if (lap > 0 && !mbar_wait(smem_addr(&freed[b * P + p]), uint32_t((lap - 1) & 1), lim)) {
            timed_out = true;  // (the wait is for row r - NB to have left this piece)
            lim = 0;
          }
          const int rest = seg_units - p * kOcPieceUnits;
          const uint32_t bytes = uint32_t(rest < kOcPieceUnits ? rest : kOcPieceUnits) * 16u;
          const uint32_t bar = smem_addr(&full[b * P + p]);
          mbar_arrive_expect_tx(bar, bytes);
          bulk_g2s(bufs + uint32_t(b) * a.buf_bytes + uint32_t(p) * kOcPieceBytes, src + int64_t(p) * kOcPieceBytes,
                   bytes, bar, drop);
          if (pf)
            oc_prefetch_l2(a.x + row_of(r + PD) * a.row_bytes + seg_start * 16 + int64_t(p) * kOcPieceBytes, bytes,
                           keep);
        }
        ring.next();
      }
      // no copy may still be in flight when the CTA exits: the last copy of every piece has landed
      for (int64_t r = M > NB ? M - NB : 0; r < M; ++r) {
        const int rb = int(r % NB);
        const uint32_t par = uint32_t((r / NB) & 1);
        for (int p = 0; p < pc; ++p)
          if (!mbar_wait(smem_addr(&full[rb * P + p]), par, a.local_wait_ns)) timed_out = true;
      }
    }
  } else if (warp == kOcPublisherWarp) {
    // Rank 0's publisher lane: the cluster state of each row as soon as the cluster's CTA states
    // have all arrived (a warp of its own, so that a publication never waits behind the exchange
    // warp's polling round trips), in row order.
    if (crank == 0 && lane == 0) {
      OcRing ring(RB);
      for (int64_t r = 0; r < M; ++r) {
        const uint32_t bar = smem_addr(&cbar[ring.idx]);
        if (!mbar_wait_cluster(bar, ring.parity(), lim)) {
          timed_out = true;
          lim = 0;
        }
        State cs = empty_state();
        for (uint32_t i = 0; i < csize; ++i) cs = merge(cs, cstate[ring.idx * kOcMaxCluster + i]);
        if (!(a.fault && cid == 0)) {
          if (local) {  // the row state into every CTA of the cluster, released by a remote arrive
            for (uint32_t q = 0; q < csize; ++q) {
              st_cluster_f32x2(map_to_rank(smem_addr(&rowst[ring.idx]), q), cs.m, cs.d);
              mbar_arrive_remote(map_to_rank(smem_addr(&row_ready[ring.idx]), q));
            }
          } else {
            oc_st_release_u64(a.pub + r * ncl + cid, oc_pack(cs));
          }
        }
        if (r + RB < M) mbar_arrive_expect_tx(bar, csize * 8u);
        ring.next();
      }
    }
  } else if (warp == kOcExchangeWarp) {
    bool abort = false;
    OcRing ring(RB);
    for (int64_t r = 0; r < (local ? 0 : M); ++r) {
      const int b = ring.idx;
      // every exit from this loop is taken by the whole warp: lane 0 alone reads the clock and
      // decides when the wait has run out (lanes that read the clock themselves could disagree at
      // the limit, and a lane that left would never reach the next full-warp collective)
      const uint64_t t0 = __shfl_sync(0xffffffffu, global_timer_ns(), 0);
      State g;
      while (true) {
        bool ready = true;
        State gg = empty_state();
        if (!abort) {
          for (uint32_t i = lane; i < ncl; i += 32) {
            const unsigned long long v = oc_ld_acquire_u64(a.pub + r * ncl + i);
            if (v == kOcUnpublished) ready = false;
            else gg = merge(gg, oc_unpack(v));
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
        rowst[b] = g;
        mbar_arrive(smem_addr(&row_ready[b]));
      }
      __syncwarp();
      ring.next();
    }
  } else {
    // ---------------- consumers ----------------
    // fold(j): row j's segment in shared-memory buffer `buf`, piece by piece as it lands, then the
    // CTA state to rank 0's slot `sb` of the state ring
    auto fold_row = [&](int64_t j, const OcRing& buf, int sb) {
      State st = empty_state();
      for (int p = 0; p < pc; ++p) {
        if (!mbar_wait(smem_addr(&full[buf.idx * P + p]), buf.parity(), lim)) {
          timed_out = true;
          lim = 0;
        }
        st = oc_fold_piece<D>(st, bufs + uint32_t(buf.idx) * a.buf_bytes + uint32_t(p) * kOcPieceBytes,
                              seg_units - p * kOcPieceUnits, tid);
      }
      const State cs = group_merge(st, wstate + (j & 1) * kOcNcw, kOcNcw, warp, lane,
                                   [] { named_barrier_sync(1, kOcNct); });
      if (tid == 0)
        oc_st_async_f32x2(map_to_rank(smem_addr(&cstate[sb * kOcMaxCluster + crank]), 0), cs.m, cs.d,
                          map_to_rank(smem_addr(&cbar[sb]), 0));
    };
    // y = e^(x - m) / d (b2 = 1 / d), or in the log mode y = (x - m) - ln d (b2 = -ln d), for the
    // four units of piece p held in q (unit p * kOcPieceUnits + i * kOcNct + tid)
    auto store_piece = [&](int64_t r, int p, const uint4 (&q)[kOcUpt], float2 nms, float2 b2) {
      unsigned char* yp = a.y + row_of(r) * a.row_bytes + (seg_start + int64_t(p) * kOcPieceUnits) * 16;
      const int rest = seg_units - p * kOcPieceUnits;
#pragma unroll
      for (int i = 0; i < kOcUpt; ++i) {
        const int u = tid + i * kOcNct;
        if (u < rest) {
          float2 f[E / 2];
          D::unpack2(q[i], f);
#pragma unroll
          for (int e = 0; e < E / 2; ++e)
            f[e] = LOG ? __fadd2_rn(__fadd2_rn(f[e], nms), b2) : __fmul2_rn(exp_diff2(f[e], nms), b2);
          st_stream16(yp + int64_t(u) * 16, D::pack2(f));
        }
      }
    };
    // row r's state (slot `sb` of the state ring), and its outputs from CTA 0 (rank 0 in local
    // mode, where the state arrives from rank 0 over DSMEM: a cluster-scope acquire, bounded by the
    // exchange limit)
    auto row_state = [&](int64_t r, const OcRing& st_ring) {
      const uint32_t bar = smem_addr(&row_ready[st_ring.idx]);
      const bool ok = local ? mbar_wait_cluster(bar, st_ring.parity(), lim == 0 ? 0 : a.exchange_wait_ns)
                            : mbar_wait(bar, st_ring.parity(), lim);
      if (!ok) {
        timed_out = true;
        lim = 0;
      }
      const State row = rowst[st_ring.idx];
      if (c == 0 && tid == 0) {
        const int64_t gr = row_of(r);
        if (a.m_out) a.m_out[gr] = row.m;
        if (a.d_out) a.d_out[gr] = row.d;
        if (a.lse_out) a.lse_out[gr] = lse_of(row);
      }
      return row;
    };

    if constexpr (!HOLD) {
      // normalise(r) from its shared-memory buffer; every piece freed right after its read
      auto normalise_row = [&](int64_t r, const OcRing& buf, const OcRing& st_ring) {
        const State row = row_state(r, st_ring);
        const float ms = safe_max(row.m);
        const float inv = LOG ? -log_norm(row).lnd : safe_inv(row.d);
        const float2 nms = make_float2(-ms, -ms), inv2 = make_float2(inv, inv);
        for (int p = 0; p < pc; ++p) {
          const uint32_t piece = bufs + uint32_t(buf.idx) * a.buf_bytes + uint32_t(p) * kOcPieceBytes;
          const int rest = seg_units - p * kOcPieceUnits;
          uint4 q[kOcUpt];
#pragma unroll
          for (int i = 0; i < kOcUpt; ++i) {
            const int u = tid + i * kOcNct;
            if (u < rest) q[i] = lds16(piece + uint32_t(u) * 16u);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_addr(&freed[buf.idx * P + p]));
          store_piece(r, p, q, nms, inv2);
        }
      };
      const int lag = NB - 1;
      OcRing fbuf(NB), fst(RB), nbuf(NB), nst(RB);
      int64_t j = 0;  // next row to fold
      for (; j < lag && j < M; ++j) {
        fold_row(j, fbuf, fst.idx);
        fbuf.next();
        fst.next();
      }
      for (int64_t r = 0; r < M; ++r) {
        if (j < M) {
          fold_row(j, fbuf, fst.idx);
          ++j;
          fbuf.next();
          fst.next();
        }
        normalise_row(r, nbuf, nst);
        nbuf.next();
        nst.next();
      }
    } else {
      // Two shared-memory buffers: rows in flight at the start of iteration r are r and r + 1
      // parked in tensor memory (slots r mod 2, r + 1 mod 2), r + 2 folded in shared-memory buffer
      // r mod 2, r + 3 landing in the other buffer.  Iteration r, piece by piece: normalise piece p
      // of row r from its slot, then park piece p of row r + 2 in its place and free that piece of
      // the buffer (row r + 4's piece is loaded there at once); then fold r + 3.  A row's state has
      // two iterations to arrive, and a buffer's load about one and a half.
      const uint32_t tmem = *tmem_slot;
      const uint32_t tlane = uint32_t(32 * (warp & 3)) << 16;
      const uint32_t tcol = uint32_t(warp >> 2) * kOcWarpCols;
      auto taddr = [&](int slot, int p) {
        return tmem + tlane + uint32_t(slot) * kOcSlotCols + tcol + uint32_t(p) * (kOcUpt * 4);
      };
      // piece p of the row in shared-memory buffer `buf` -> tensor-memory slot, the piece freed once read
      auto park_piece = [&](const OcRing& buf, int slot, int p) {
        const uint32_t piece = bufs + uint32_t(buf.idx) * a.buf_bytes + uint32_t(p) * kOcPieceBytes;
        const int rest = seg_units - p * kOcPieceUnits;
        uint4 q[kOcUpt];
#pragma unroll
        for (int i = 0; i < kOcUpt; ++i) {
          const int u = tid + i * kOcNct;
          q[i] = u < rest ? lds16(piece + uint32_t(u) * 16u) : make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();  // (tensor-memory accesses are warp-wide)
        oc_tmem_st16(taddr(slot, p), q);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&freed[buf.idx * P + p]));
      };
      OcRing fbuf(NB), fst(RB);  // next row to fold: its buffer and state slot
      OcRing pbuf(NB);           // next row to park: its buffer
      OcRing nst(RB);            // next row to normalise: its state slot
      int64_t jf = 0, jp = 0;    // next rows to fold and to park
      auto fold_next = [&]() {
        if (jf < M) {
          fold_row(jf, fbuf, fst.idx);
          ++jf;
          fbuf.next();
          fst.next();
        }
      };
      auto park_next = [&]() {  // a whole row
        if (jp < M) {
          for (int p = 0; p < pc; ++p) park_piece(pbuf, int(jp & 1), p);
          oc_tmem_wait_st();
          ++jp;
          pbuf.next();
        }
      };
      auto normalise_parked = [&](int64_t r, bool park_behind) {
        const int slot = int(r & 1);
        const State row = row_state(r, nst);
        nst.next();
        const float ms = safe_max(row.m);
        const float inv = LOG ? -log_norm(row).lnd : safe_inv(row.d);
        const float2 nms = make_float2(-ms, -ms), inv2 = make_float2(inv, inv);
        for (int p = 0; p < pc; ++p) {
          uint4 q[kOcUpt];
          __syncwarp();
          oc_tmem_ld16(taddr(slot, p), q);
          oc_tmem_wait_ld();
          store_piece(r, p, q, nms, inv2);
          if (park_behind) park_piece(pbuf, slot, p);
        }
        if (park_behind) {
          oc_tmem_wait_st();
          ++jp;
          pbuf.next();
        }
      };
      if (NB >= 2) {
        fold_next();  // row 0
        park_next();
        fold_next();  // row 1
        park_next();
        fold_next();  // row 2
        for (int64_t r = 0; r < M; ++r) {
          normalise_parked(r, jp < M);  // row jp = r + 2 follows row r into its slot, piece by piece
          fold_next();                  // row r + 3
        }
      } else {
        // One shared-memory buffer (segments of up to 128 KB).  Iteration r: park r + 1 in the slot
        // row r - 1 left (its buffer is then loaded with row r + 2), normalise r, fold r + 2.
        fold_next();  // row 0
        park_next();
        fold_next();  // row 1
        for (int64_t r = 0; r < M; ++r) {
          park_next();  // row r + 1
          normalise_parked(r, false);
          fold_next();  // row r + 2
        }
      }
      // every consumer is done with tensor memory before it is released
      oc_tc_fence_before();
      named_barrier_sync(1, kOcNct);
      oc_tc_fence_after();
      if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kOcTmemCols));
    }
  }
  if (timed_out) atomicOr(a.status, kStatusTimeout);
  __syncwarp();
  oc_cluster_sync_all();
}

using OnchipKernel = void (*)(OnchipArgs);

template <bool LOG>
OnchipKernel onchip_kernel_of(int dtype, bool hold) {
  if (hold) return dtype == 0 ? k_splitrow_onchip<F32, true, LOG> : dtype == 1 ? k_splitrow_onchip<BF16, true, LOG>
                                                                              : k_splitrow_onchip<F16, true, LOG>;
  return dtype == 0 ? k_splitrow_onchip<F32, false, LOG> : dtype == 1 ? k_splitrow_onchip<BF16, false, LOG>
                                                                      : k_splitrow_onchip<F16, false, LOG>;
}
// The log-softmax instances (local mode only) use the registers and shared memory of the others,
// so the residency plans below, taken with the softmax instance, hold for them too.
OnchipKernel onchip_kernel(int dtype, bool hold, bool log = false) {
  return log ? onchip_kernel_of<true>(dtype, hold) : onchip_kernel_of<false>(dtype, hold);
}

// Cluster size and count for the largest shared-memory footprint (one CTA per SM), per device and
// element type.  The footprint of a launch depends on the row length, but the residency of one
// CTA per SM does not, so the plan is taken once at the largest size.
struct OnchipPlan {
  bool ok = false;
  int cluster = 0;
  int clusters = 0;
};

std::mutex g_oc_mutex;
OnchipPlan g_oc_plan[64][3];
bool g_oc_ready[64][3];

OnchipPlan onchip_plan(int dtype, const DeviceInfo& dev) {
  std::lock_guard<std::mutex> lock(g_oc_mutex);
  if (dev.device >= 0 && dev.device < 64 && g_oc_ready[dev.device][dtype]) return g_oc_plan[dev.device][dtype];
  OnchipPlan best;
  if (dev.cluster_launch) {
    const size_t smem = size_t(dev.max_smem_per_block_optin);
    OnchipKernel fn = onchip_kernel(dtype, false);
    if (cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) == cudaSuccess) {
      for (int cs : {8, 4, 2}) {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3(kOcThreads);
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
        }
      }
    } else {
      cudaGetLastError();
    }
  }
  if (dev.device >= 0 && dev.device < 64) {
    g_oc_plan[dev.device][dtype] = best;
    g_oc_ready[dev.device][dtype] = true;
  }
  return best;
}

struct OnchipShape {
  bool ok = false;
  bool hold = false;  // segments parked in tensor memory (one or two shared-memory buffers)
  bool local = false;
  int nb = 0, rb = 0, pieces = 0;
  uint32_t buf_bytes = 0;
  size_t smem = 0;
  int G = 0, cluster = 0;  // CTAs launched, CTAs per cluster
};

// Buffers for segments of up to seg_max units: as many shared-memory buffers as fit (up to 8); with
// two, folded segments are parked in tensor memory (two slots of kOcWarpCols columns per warp), and
// with one too when `one_buffer` allows it.  False when the segments do not fit.
bool segment_buffers(int64_t seg_max, int64_t rows, size_t cap, bool one_buffer, OnchipShape* s) {
  const int64_t pieces = (seg_max + kOcPieceUnits - 1) / kOcPieceUnits;
  if (pieces > kOcMaxPieces) return false;
  const int64_t buf = (seg_max * 16 + 127) / 128 * 128;
  const bool parkable = pieces * kOcUpt * 4 <= int64_t(kOcWarpCols);
  int nb = kOcMaxBufs;
  while (nb >= 1 && size_t(nb) * size_t(buf) + onchip_tail_bytes(nb, nb < 3 ? 4 : nb, int(pieces)) > cap) --nb;
  if (nb >= 3) {
    // fold NB - 1 rows ahead
    if (rows < nb) nb = int(rows < 2 ? 2 : rows);
    s->hold = false;
    s->rb = nb;
  } else if (parkable && (nb == 2 || (nb == 1 && one_buffer))) {
    // park folded segments in tensor memory (rows r .. r + 3 in flight with two buffers, r .. r + 2
    // with one)
    s->hold = true;
    s->rb = 4;
  } else {
    return false;
  }
  s->nb = nb;
  s->pieces = int(pieces);
  s->buf_bytes = uint32_t(buf);
  s->smem = size_t(nb) * size_t(buf) + onchip_tail_bytes(nb, s->rb, int(pieces));
  return true;
}

// Split mode: one row over every CTA of the grid.
OnchipShape onchip_shape(const RowProblem& p, const DeviceInfo& dev) {
  OnchipShape s;
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  if (row_bytes % 16 != 0 || p.log_out) return s;
  const OnchipPlan plan = onchip_plan(p.dtype, dev);
  if (!plan.ok) return s;
  const int64_t G = int64_t(plan.cluster) * plan.clusters;
  const int64_t units = row_bytes / 16;
  if (units < G * 64) return s;  // rows this short belong to the one-read row kernels
  const int64_t seg_max = (units + G - 1) / G;
  if (!segment_buffers(seg_max, p.M, size_t(dev.max_smem_per_block_optin), false, &s)) return s;
  s.ok = true;
  s.G = int(G);
  s.cluster = plan.cluster;
  return s;
}

// Local mode: resident clusters of 2, 4, 8 and 16 CTAs (one CTA per SM), per device and element type.
// Clusters of 16 are not used (measured, 300 x 2 MiB fp32 rows held on chip by clusters of 16:
// 305 us against 239 us for the cluster-row two passes).
constexpr int kOcLocalSizes[4] = {2, 4, 8, 16};
constexpr int kOcLocalMaxCluster = 8;
struct LocalPlan {
  int n[4] = {0, 0, 0, 0};
};
std::mutex g_ocl_mutex;
LocalPlan g_ocl[64][3];
bool g_ocl_ready[64][3];

LocalPlan local_plan(int dtype, const DeviceInfo& dev) {
  std::lock_guard<std::mutex> lock(g_ocl_mutex);
  const bool cache = dev.device >= 0 && dev.device < 64;
  if (cache && g_ocl_ready[dev.device][dtype]) return g_ocl[dev.device][dtype];
  LocalPlan lp;
  if (dev.cluster_launch) {
    const size_t smem = size_t(dev.max_smem_per_block_optin);
    for (bool hold : {false, true}) {  // both instances may launch clusters of 16
      OnchipKernel fn = onchip_kernel(dtype, hold);
      if (cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess ||
          cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
        cudaGetLastError();
    }
    OnchipKernel fn = onchip_kernel(dtype, false);
    for (int i = 0; i < 4; ++i) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = kOcLocalSizes[i];
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(kOcLocalSizes[i]);
      cfg.blockDim = dim3(kOcThreads);
      cfg.dynamicSmemBytes = smem;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, (const void*)fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
      }
      lp.n[i] = n;
    }
  }
  if (cache) {
    g_ocl[dev.device][dtype] = lp;
    g_ocl_ready[dev.device][dtype] = true;
  }
  return lp;
}

// Local mode: the smallest cluster whose segments fit on chip (one shared-memory buffer with
// tensor-memory parking at the least), as many resident clusters as the occupancy query reports.
OnchipShape onchip_local_shape(const RowProblem& p, const DeviceInfo& dev) {
  OnchipShape s;
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  if (row_bytes % 16 != 0 || p.y == nullptr || p.labels || p.loss) return s;
  if ((p.x_pitch && p.x_pitch != row_bytes) || (p.y_pitch && p.y_pitch != row_bytes) || p.scale != 1.f) return s;
  const int64_t units = row_bytes / 16;
  const LocalPlan lp = local_plan(p.dtype, dev);
  for (int i = 0; i < 4; ++i) {
    const int cs = kOcLocalSizes[i];
    if (cs > kOcLocalMaxCluster || lp.n[i] < 1 || units < int64_t(cs) * 64) continue;
    const int64_t clusters = p.M < lp.n[i] ? p.M : lp.n[i];
    const int64_t rows = (p.M + clusters - 1) / clusters;  // rows of the busiest cluster
    if (!segment_buffers((units + cs - 1) / cs, rows, size_t(dev.max_smem_per_block_optin), true, &s)) continue;
    s.ok = true;
    s.local = true;
    s.G = int(clusters * cs);
    s.cluster = cs;
    return s;
  }
  return s;
}

cudaError_t launch_onchip(const RowProblem& p, const DeviceInfo& dev, const OnchipShape& s, unsigned long long* pub) {
  OnchipKernel fn = onchip_kernel(p.dtype, s.hold, p.log_out);
  cudaError_t err = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(s.smem));
  if (err != cudaSuccess) return err;
  if (s.cluster > 8 &&
      (err = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != cudaSuccess)
    return err;
  OnchipArgs a;
  a.x = static_cast<const unsigned char*>(p.x);
  a.y = static_cast<unsigned char*>(p.y);
  a.m_out = p.m_out;
  a.d_out = p.d_out;
  a.lse_out = p.lse_out;
  a.M = p.M;
  a.row_bytes = p.N * elem_bytes(p.dtype);
  a.units = a.row_bytes / 16;
  a.nb = s.nb;
  a.rb = s.rb;
  a.pieces = s.pieces;
  a.buf_bytes = s.buf_bytes;
  a.pub = pub;
  a.status = dev.status;
  a.local_wait_ns = local_wait_limit_ns();
  a.exchange_wait_ns = exchange_wait_limit_ns();
  a.fault = debug_fault();
  a.local = s.local ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = s.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(s.G);
  cfg.blockDim = dim3(kOcThreads);
  cfg.dynamicSmemBytes = s.smem;
  cfg.stream = p.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, a);
}

}  // namespace

bool splitrow_onchip_fits(const RowProblem& p, const DeviceInfo& dev) { return onchip_shape(p, dev).ok; }

cudaError_t launch_splitrow_onchip(const RowProblem& p, const DeviceInfo& dev, unsigned long long* pub) {
  const OnchipShape s = onchip_shape(p, dev);
  if (!s.ok) return cudaErrorInvalidConfiguration;
  return launch_onchip(p, dev, s, pub);
}

bool clusterrow_onchip_fits(const RowProblem& p, const DeviceInfo& dev) { return onchip_local_shape(p, dev).ok; }

cudaError_t launch_clusterrow_onchip(const RowProblem& p, const DeviceInfo& dev) {
  const OnchipShape s = onchip_local_shape(p, dev);
  if (!s.ok) return cudaErrorInvalidConfiguration;
  return launch_onchip(p, dev, s, nullptr);
}

int splitrow_onchip_clusters(const RowProblem& p, const DeviceInfo& dev) {
  const OnchipShape s = onchip_shape(p, dev);
  return s.ok ? s.G / s.cluster : 0;
}

cudaError_t launch_splitrow_onchip_pooled(const RowProblem& p, const DeviceInfo& dev) {
  const int ncl = splitrow_onchip_clusters(p, dev);
  if (ncl <= 0) return cudaErrorInvalidConfiguration;
  // one 64-bit publication slot per (row, cluster), stream-ordered, all ones until published
  const size_t pub_bytes = size_t(p.M) * ncl * sizeof(unsigned long long);
  void* scratch = nullptr;
  cudaError_t err = cudaMallocAsync(&scratch, pub_bytes, p.stream);
  if (err != cudaSuccess) return err;
  err = cudaMemsetAsync(scratch, 0xFF, pub_bytes, p.stream);
  if (err == cudaSuccess) err = launch_splitrow_onchip(p, dev, static_cast<unsigned long long*>(scratch));
  const cudaError_t ferr = cudaFreeAsync(scratch, p.stream);
  return err != cudaSuccess ? err : ferr;
}

}  // namespace rwo
