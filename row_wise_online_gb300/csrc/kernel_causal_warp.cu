// kernel_causal_warp.cu -- softmax of causally masked rows that never reads the masked entries.
//
// In causal attention a query at position q only sees keys 0..q; the scores of the later keys
// are -inf, their exponentials 0, so they change neither m nor d (the recurrence of
// "5.2 CUDA Online Softmax 实现优化" §2.1 with e^(-inf) = 0), and "Softmax 数值稳定性与
// IO-Aware Attention" §八 skips such fully masked blocks.  Row r of the score matrix therefore
// only has a live prefix of L_r = clamp(r % q_period + 1 + key_offset, 0, N) entries.
// This kernel folds and normalises that prefix and writes y = 0 for the rest without reading it:
// on a square causal mask it reads about half of x.
//
// Same shape as the warp-per-row one-read kernel (one warp per row, the row staged in shared
// memory by a bulk copy issued by lane 0, two passes over shared memory, 16-byte streaming
// stores), with two differences that come from the rows' unequal live lengths:
//
//  * each warp owns a byte ring instead of fixed row slots: live prefixes are packed back to back
//    (first in first out, wrapping to offset 0; up to kRingRows rows in flight, one mbarrier
//    each), so the bytes a warp has in flight stay near the ring size however short the rows;
//  * the fold and the normalisation run over whole steps inside the live prefix without any
//    bounds test, one checked step for the vector that straddles L_r (its dead entries are set
//    to -inf in registers), and a store-only loop for the zeros.
// Adds and multiplies use the packed f32x2 instructions (each half rounded as the scalar
// operation).  Every wait is bounded (%globaltimer).
#include <type_traits>

#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

struct CausalArgs {
  const unsigned char* x;
  unsigned char* y;
  float* m_out;
  float* d_out;
  float* lse_out;
  int64_t M;
  int64_t N;
  uint32_t row_bytes;
  uint32_t ring_bytes;  // per warp
  unsigned* status;
  uint64_t wait_ns;
  int64_t q_period;    // row r keeps its first clamp(r % q_period + 1 + key_offset, 0, N) entries;
  int64_t key_offset;  // the rest count as -inf and are never read
};

constexpr int kStep = 4;      // 16-byte vectors per lane per step
constexpr int kRingRows = 8;  // rows in flight per warp at most (one mbarrier each)

template <class D, int VPL>
__global__ void __launch_bounds__(512, 1) k_causal_warp(CausalArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int E = D::kVec;
  constexpr int K = kRingRows;
  constexpr int kStepUnits = kStep * 32;  // vectors per warp step
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t RB = a.ring_bytes;
  unsigned char* ring = smem + size_t(warp) * RB;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(W) * RB) + size_t(warp) * K;
  uint32_t* roff = reinterpret_cast<uint32_t*>(smem + size_t(W) * RB + size_t(W) * K * sizeof(uint64_t)) +
                   size_t(warp) * K;  // ring offset of each row in flight

  if (lane == 0) {
    for (int i = 0; i < K; ++i) mbar_init(smem_addr(&full[i]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int64_t gw = int64_t(blockIdx.x) * W + warp;
  const int64_t GW = int64_t(gridDim.x) * W;
  const int nrows = a.M > gw ? int((a.M - 1 - gw) / GW + 1) : 0;  // the host keeps this below 2^31
  const int nunits = int(a.N / E);
  const uint64_t pol = policy_evict_first();

  // Position r % q_period of the warp's rows, stepped without a division per row; one copy
  // follows the rows being issued, one the rows being processed.
  struct QPos {
    int64_t q, step, period;
    __device__ void next() {
      q += step;
      if (q >= period) q -= period;
    }
  };
  QPos q_iss{gw % a.q_period, GW % a.q_period, a.q_period};
  QPos q_cur = q_iss;
  auto live_len = [&](const QPos& qp) -> int {  // at most N <= 8192 here
    const int64_t L = qp.q + 1 + a.key_offset;
    return int(L < 0 ? 0 : (L > a.N ? a.N : L));
  };

  // Ring placement: every lane computes the same offsets, lane 0 writes them and issues the copy.
  int issued = 0;
  uint32_t head = 0;  // end of the last issued row
  auto refill = [&](int done) {
    while (issued < nrows && issued - done < K) {
      const int lu = (live_len(q_iss) + E - 1) / E;
      const uint32_t b = uint32_t(lu > 0 ? lu : 1) * 16u;  // at least one vector: the barrier completes
      uint32_t off;
      if (issued == done) {
        off = 0;  // ring empty
      } else {
        const uint32_t tail = roff[done % K];  // start of the oldest row still in use
        if (head > tail) {                     // in use: [tail, head)
          if (head + b <= RB) off = head;
          else if (b <= tail) off = 0;
          else break;
        } else {  // in use: [tail, RB) and [0, head); the ring is full when head == tail
          if (head + b <= tail) off = head;
          else break;
        }
      }
      if (lane == 0) {
        const int i = issued % K;
        roff[i] = off;
        mbar_arrive_expect_tx(smem_addr(&full[i]), b);
        bulk_g2s(smem_addr(ring + off), a.x + (gw + int64_t(issued) * GW) * a.row_bytes, b, smem_addr(&full[i]),
                 pol);
      }
      head = off + b;
      ++issued;
      q_iss.next();
    }
    __syncwarp();  // the offsets written by lane 0 are visible to the warp
  };
  refill(0);

  bool timed_out = false;
  for (int j = 0; j < nrows; ++j) {
    const int ib = j % K;
    if (!mbar_wait(smem_addr(&full[ib]), uint32_t((j / K) & 1), a.wait_ns)) timed_out = true;
    const uint32_t slot = smem_addr(ring + roff[ib]);
    const int64_t row = gw + int64_t(j) * GW;
    const int L = live_len(q_cur);        // live elements
    const int lunits = (L + E - 1) / E;   // vectors read
    const int nfull = (L / E) / kStepUnits;  // steps wholly inside the live prefix

    // pass 1: online fold of the live prefix, one rescale per step
    State st = empty_state();
    auto fold_step = [&](int k0, auto checked) {
      uint4 q[kStep];
#pragma unroll
      for (int i = 0; i < kStep; ++i) {
        const int u = lane + (k0 + i) * 32;
        if constexpr (decltype(checked)::value) {
          q[i] = u < lunits ? lds16(slot + uint32_t(u) * 16u)
                            : make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
          const int keep = L - u * E;  // the straddling vector keeps only its live entries
          if (keep > 0 && keep < E) q[i] = mask_tail<D>(q[i], keep);
        } else {
          q[i] = lds16(slot + uint32_t(u) * 16u);
        }
      }
      float mu = -INFINITY;
#pragma unroll
      for (int i = 0; i < kStep; ++i) mu = fmaxf(mu, D::vmax(q[i]));
      const float m_new = fmaxf(st.m, mu);
      const float ms = safe_max(m_new);
      const float2 nms = make_float2(-ms, -ms);
      float2 acc = make_float2(0.f, 0.f);  // two partial sums, one per half of the pairs
#pragma unroll
      for (int i = 0; i < kStep; ++i) {
        float2 f[E / 2];
        D::unpack2(q[i], f);
#pragma unroll
        for (int e = 0; e < E / 2; ++e) acc = __fadd2_rn(acc, exp_diff2(f[e], nms));
      }
      st.d = __fadd_rn(__fmul_rn(st.d, exp_diff(st.m, ms)), __fadd_rn(acc.x, acc.y));
      st.m = m_new;
    };
#pragma unroll 1
    for (int s = 0; s < nfull; ++s) fold_step(s * kStep, std::false_type{});
    if (nfull * kStepUnits < lunits) fold_step(nfull * kStep, std::true_type{});  // at most one left
    st = warp_merge(st);

    // pass 2: normalise the live prefix, zeros after it
    const float ms = safe_max(st.m);
    const float inv = safe_inv(st.d);
    const float2 nms = make_float2(-ms, -ms), inv2 = make_float2(inv, inv);
    unsigned char* yr = a.y + row * a.row_bytes;
    auto norm_step = [&](int k0, auto checked) {
      constexpr bool kChecked = decltype(checked)::value;
      uint4 q[kStep];
#pragma unroll
      for (int i = 0; i < kStep; ++i) {
        const int u = lane + (k0 + i) * 32;
        if (!kChecked || u < lunits) q[i] = lds16(slot + uint32_t(u) * 16u);
      }
#pragma unroll
      for (int i = 0; i < kStep; ++i) {
        const int u = lane + (k0 + i) * 32;
        if (!kChecked || u < lunits) {
          if constexpr (kChecked) {
            const int keep = L - u * E;
            if (keep < E) q[i] = mask_tail<D>(q[i], keep);  // -inf -> y = 0 there
          }
          float2 f[E / 2];
          D::unpack2(q[i], f);
#pragma unroll
          for (int e = 0; e < E / 2; ++e) f[e] = __fmul2_rn(exp_diff2(f[e], nms), inv2);
          st_stream16(yr + int64_t(u) * 16, D::pack2(f));
        } else if (u < nunits) {
          st_stream16(yr + int64_t(u) * 16, make_uint4(0u, 0u, 0u, 0u));  // masked: y = 0, x not read
        }
      }
    };
#pragma unroll 1
    for (int s = 0; s < nfull; ++s) norm_step(s * kStep, std::false_type{});
    int k0 = nfull * kStep;
    if (k0 * 32 < lunits) {
      norm_step(k0, std::true_type{});
      k0 += kStep;
    }
#pragma unroll 1
    for (; k0 * 32 < nunits; k0 += kStep) {  // wholly masked: zeros only
#pragma unroll
      for (int i = 0; i < kStep; ++i) {
        const int u = lane + (k0 + i) * 32;
        if (u < nunits) st_stream16(yr + int64_t(u) * 16, make_uint4(0u, 0u, 0u, 0u));
      }
    }
    if (lane == 0) {
      if (a.m_out) a.m_out[row] = st.m;
      if (a.d_out) a.d_out[row] = st.d;
      if (a.lse_out) a.lse_out[row] = lse_of(st);
    }
    // hand row j's bytes back (generic reads before the async-proxy refill) and refill
    fence_proxy_async_smem();
    __syncwarp();
    q_cur.next();
    refill(j + 1);
  }
  if (timed_out && lane == 0) atomicOr(a.status, kStatusTimeout);
}

using CausalKernel = void (*)(CausalArgs);

struct CausalConfig {
  int vpl;  // 16-byte vectors per lane (row capacity 32 * vpl vectors)
  CausalKernel fn[3];  // [dtype]
};

template <int VPL>
constexpr CausalConfig causal_cfg() {
  return CausalConfig{VPL, {k_causal_warp<F32, VPL>, k_causal_warp<BF16, VPL>, k_causal_warp<F16, VPL>}};
}

const CausalConfig kCausalCfg[] = {causal_cfg<4>(), causal_cfg<8>(), causal_cfg<16>(), causal_cfg<32>()};

struct CausalPlan {
  const CausalConfig* cfg = nullptr;
  int warps = 0;            // per CTA
  uint32_t ring_bytes = 0;  // per warp
  size_t smem = 0;
};

constexpr uint32_t kRingAlign = 128;
constexpr int64_t kMaxRowBytes = 16384;

// A ring of three whole rows per warp (four for rows of at most 2 KB); as many warps as ~200 KB
// of shared memory per SM holds, at most 16 per CTA, and CTAs of 4 warps (two per SM) for rows
// above 4 KiB, as for the warp-per-row kernel (measured on the 524,288 x 4096 bf16 causal rows:
// 1.022 against 1.031 ms with one CTA of 8 warps per SM; CTAs of 2 warps 1.026, of 6 1.371).
CausalPlan plan_causal(const RowProblem& p, const DeviceInfo& dev) {
  CausalPlan plan;
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  if (row_bytes % 16 != 0 || row_bytes > kMaxRowBytes) return plan;
  if (p.M / dev.sm_count >= INT32_MAX) return plan;  // rows per warp are counted in 32 bits
  const int64_t units = row_bytes / 16;
  const CausalConfig* cfg = nullptr;
  for (const CausalConfig& c : kCausalCfg)
    if (units <= int64_t(32) * c.vpl) {
      cfg = &c;
      break;
    }
  if (!cfg) return plan;
  const uint32_t rows = row_bytes <= 2048 ? 4 : 3;
  const uint32_t ring = uint32_t((rows * row_bytes + kRingAlign - 1) / kRingAlign * kRingAlign);
  const size_t per_warp = size_t(ring) + kRingRows * (sizeof(uint64_t) + sizeof(uint32_t));
  const size_t budget = size_t(dev.max_smem_per_sm) > 32768 ? size_t(dev.max_smem_per_sm) - 28672 : 0;
  int warps_sm = int(budget / per_warp);
  if (warps_sm > 32) warps_sm = 32;
  if (warps_sm < 1) return plan;
  const int cta_warps = row_bytes > 4096 ? 4 : 16;
  int warps = warps_sm < cta_warps ? warps_sm : cta_warps;
  if (size_t(warps) * per_warp > size_t(dev.max_smem_per_block_optin))
    warps = int(dev.max_smem_per_block_optin / per_warp);
  if (warps < 1) return plan;
  plan.cfg = cfg;
  plan.warps = warps;
  plan.ring_bytes = ring;
  plan.smem = size_t(warps) * per_warp;
  return plan;
}

}  // namespace

bool causal_warp_fits(const RowProblem& p, const DeviceInfo& dev) { return plan_causal(p, dev).cfg != nullptr; }

cudaError_t launch_causal_warp(const RowProblem& p, const DeviceInfo& dev, int64_t q_period, int64_t key_offset) {
  const CausalPlan plan = plan_causal(p, dev);
  if (!plan.cfg || q_period < 1) return cudaErrorInvalidValue;
  CausalKernel fn = plan.cfg->fn[p.dtype];
  cudaError_t err = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(plan.smem));
  if (err != cudaSuccess) return err;
  const int threads = plan.warps * 32;
  int occ = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, (const void*)fn, threads, plan.smem);
  if (err != cudaSuccess) return err;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t want = (p.M + plan.warps - 1) / plan.warps;
  const int64_t cap = int64_t(dev.sm_count) * occ;
  const int grid = int(want < cap ? want : cap);
  CausalArgs a{static_cast<const unsigned char*>(p.x), static_cast<unsigned char*>(p.y), p.m_out, p.d_out,
               p.lse_out, p.M, p.N, uint32_t(p.N * elem_bytes(p.dtype)), plan.ring_bytes, dev.status,
               local_wait_limit_ns(), q_period, key_offset};
  fn<<<grid, threads, plan.smem, p.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace rwo
