// kernel_oneread_warp.cu -- one-read softmax for short rows: one warp per row, rows staged in
// shared memory by bulk copies.
//
// "5.2 CUDA Online Softmax 实现优化" §6 keeps the row on chip so that x is read from HBM once and
// y written once; §4.3's warp-shuffle merge finishes the row when one warp owns it.  For rows of
// up to 16 KB this kernel gives every warp its own small ring of row slots in shared memory:
//
//  * lane 0 of each warp issues cp.async.bulk global -> shared for the warp's next rows
//    (completion counted in bytes on a per-slot mbarrier), so every warp keeps S - 1 rows of
//    HBM reads in flight while it works on one;
//  * the warp folds its row from shared memory into per-lane (m, d) states, four 16-byte vectors
//    at a time (the online recurrence with one rescale per step, one exponential per element),
//    merges them with a butterfly, then normalises in a second pass over shared memory and
//    writes y with 16-byte streaming stores;
//  * the slot is handed back (proxy fence, warp sync) and lane 0 refills it with the row S
//    positions ahead.
// There is no block-level synchronisation at all: warps run independently.  Persistent grid:
// global warp w handles rows w, w + (total warps), ...  Every wait is bounded (%globaltimer).
#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

struct WarpArgs {
  const unsigned char* x;
  unsigned char* y;
  float* m_out;
  float* d_out;
  float* lse_out;
  int64_t M;
  int64_t N;
  uint32_t row_bytes;
  uint32_t slot_bytes;
  int slots;  // per warp
  unsigned* status;
  uint64_t wait_ns;
};

constexpr int kStep = 4;  // 16-byte vectors per lane in flight per step

template <class D, int VPL>
__global__ void __launch_bounds__(512) k_oneread_warp(WarpArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int E = D::kVec;
  const int W = blockDim.x >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = a.slots;
  unsigned char* my_slots = smem + size_t(warp) * S * a.slot_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(W) * S * a.slot_bytes) + size_t(warp) * S;

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(smem_addr(&full[s]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  const int64_t gw = int64_t(blockIdx.x) * W + warp;
  const int64_t GW = int64_t(gridDim.x) * W;
  const int64_t nrows = a.M > gw ? (a.M - 1 - gw) / GW + 1 : 0;
  const int64_t nunits = a.N / E;
  const uint64_t pol = policy_evict_first();

  auto issue = [&](int64_t j) {  // lane 0: load row j of this warp into slot j % S
    const int s = int(j % S);
    const uint32_t bar = smem_addr(&full[s]);
    mbar_arrive_expect_tx(bar, a.row_bytes);
    bulk_g2s(smem_addr(my_slots + size_t(s) * a.slot_bytes), a.x + (gw + j * GW) * a.row_bytes, a.row_bytes, bar,
             pol);
  };
  if (lane == 0)
    for (int64_t j = 0; j < S && j < nrows; ++j) issue(j);

  bool timed_out = false;
  for (int64_t j = 0; j < nrows; ++j) {
    const int s = int(j % S);
    if (!mbar_wait(smem_addr(&full[s]), uint32_t((j / S) & 1), a.wait_ns)) timed_out = true;
    const uint32_t slot = smem_addr(my_slots + size_t(s) * a.slot_bytes);
    const int64_t row = gw + j * GW;

    // pass 1: online fold, one rescale per step of kStep vectors
    State st = empty_state();
#pragma unroll
    for (int k0 = 0; k0 < VPL; k0 += kStep) {
      uint4 q[kStep];
#pragma unroll
      for (int i = 0; i < kStep; ++i) {
        const int u = lane + (k0 + i) * 32;
        q[i] = u < nunits ? lds16(slot + uint32_t(u) * 16u)
                          : make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
      }
      float mu = -INFINITY;
#pragma unroll
      for (int i = 0; i < kStep; ++i) mu = fmaxf(mu, D::vmax(q[i]));
      const float m_new = fmaxf(st.m, mu);
      const float ms = safe_max(m_new);
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < kStep; ++i) {
        float f[E];
        D::unpack(q[i], f);
#pragma unroll
        for (int e = 0; e < E; ++e) acc += exp_diff(f[e], ms);
      }
      st.d = __fadd_rn(__fmul_rn(st.d, exp_diff(st.m, ms)), acc);
      st.m = m_new;
    }
    st = warp_merge(st);

    // pass 2: normalise from shared memory, 16-byte streaming stores
    const float ms = safe_max(st.m);
    const float inv = safe_inv(st.d);
    unsigned char* yr = a.y + row * a.row_bytes;
#pragma unroll
    for (int k0 = 0; k0 < VPL; k0 += kStep) {
      uint4 q[kStep];
#pragma unroll
      for (int i = 0; i < kStep; ++i) {
        const int u = lane + (k0 + i) * 32;
        if (u < nunits) q[i] = lds16(slot + uint32_t(u) * 16u);
      }
#pragma unroll
      for (int i = 0; i < kStep; ++i) {
        const int u = lane + (k0 + i) * 32;
        if (u < nunits) {
          float f[E];
          D::unpack(q[i], f);
#pragma unroll
          for (int e = 0; e < E; ++e) f[e] = __fmul_rn(exp_diff(f[e], ms), inv);
          st_stream16(yr + int64_t(u) * 16, D::pack(f));
        }
      }
    }
    if (lane == 0) {
      if (a.m_out) a.m_out[row] = st.m;
      if (a.d_out) a.d_out[row] = st.d;
      if (a.lse_out) a.lse_out[row] = lse_of(st);
    }
    // hand the slot back: generic reads before the async-proxy refill
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && j + S < nrows) issue(j + S);
  }
  if (timed_out && lane == 0) atomicOr(a.status, kStatusTimeout);
}

using WarpKernel = void (*)(WarpArgs);

struct WarpConfig {
  int vpl;  // 16-byte vectors per lane (row capacity 32 * vpl vectors)
  WarpKernel fn[3];  // [dtype]
};

template <int VPL>
constexpr WarpConfig warp_cfg() {
  return WarpConfig{VPL, {k_oneread_warp<F32, VPL>, k_oneread_warp<BF16, VPL>, k_oneread_warp<F16, VPL>}};
}

const WarpConfig kWarpCfg[] = {warp_cfg<4>(), warp_cfg<8>(), warp_cfg<16>(), warp_cfg<32>()};

struct WarpPlan {
  const WarpConfig* cfg = nullptr;
  int warps = 0;  // per CTA
  int slots = 0;  // per warp
  uint32_t slot_bytes = 0;
  size_t smem = 0;
};

constexpr uint32_t kWarpSlotAlign = 128;
constexpr int64_t kWarpMaxRowBytes = 16384;

// Four slots per warp for rows of at most 2 KB, three above; as many warps as ~200 KB of shared
// memory per SM holds, at most 16 per CTA -- and for rows above 4 KiB CTAs of 4 warps, several per
// SM (measured, bf16, TB/s with CTAs of 16 / 8 / 4 warps: 8 KiB rows 6.53 / 6.53 / 6.63 -- the
// 524,288 x 4096 workload 1.298 -> 1.279 ms --, 6 KiB 5.92 / 5.34 / 6.27; but 4 KiB 5.94 / 5.87 /
// 5.76 and 3 KiB 6.07 / 6.02 / 5.88).
WarpPlan plan_warp(const RowProblem& p, const DeviceInfo& dev) {
  WarpPlan plan;
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  if (row_bytes % 16 != 0 || row_bytes > kWarpMaxRowBytes) return plan;
  const int64_t units = row_bytes / 16;
  const WarpConfig* cfg = nullptr;
  for (const WarpConfig& c : kWarpCfg)
    if (units <= int64_t(32) * c.vpl) {
      cfg = &c;
      break;
    }
  if (!cfg) return plan;
  const uint32_t slot = uint32_t((row_bytes + kWarpSlotAlign - 1) / kWarpSlotAlign * kWarpSlotAlign);
  const int slots = row_bytes <= 2048 ? 4 : 3;
  const size_t per_warp = size_t(slots) * (slot + sizeof(uint64_t));
  const size_t budget = size_t(dev.max_smem_per_sm) > 32768 ? size_t(dev.max_smem_per_sm) - 28672 : 0;
  int warps_sm = int(budget / per_warp);
  if (warps_sm > 32) warps_sm = 32;
  if (warps_sm < 1) return plan;
  const int cta_warps = row_bytes > 4096 ? 4 : 16;
  int warps = warps_sm < cta_warps ? warps_sm : cta_warps;
  if (size_t(warps) * per_warp > size_t(dev.max_smem_per_block_optin)) warps = int(dev.max_smem_per_block_optin / per_warp);
  if (warps < 1) return plan;
  plan.cfg = cfg;
  plan.warps = warps;
  plan.slots = slots;
  plan.slot_bytes = slot;
  plan.smem = size_t(warps) * per_warp;
  return plan;
}

}  // namespace

bool oneread_warp_fits(const RowProblem& p, const DeviceInfo& dev) { return plan_warp(p, dev).cfg != nullptr; }

cudaError_t launch_oneread_warp(const RowProblem& p, const DeviceInfo& dev) {
  const WarpPlan plan = plan_warp(p, dev);
  if (!plan.cfg) return cudaErrorInvalidValue;
  WarpKernel fn = plan.cfg->fn[p.dtype];
  cudaError_t err = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(plan.smem));
  if (err != cudaSuccess) return err;
  const int threads = plan.warps * 32;
  int occ = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, (const void*)fn, threads, plan.smem);
  if (err != cudaSuccess) return err;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t rows_per_cta = plan.warps;
  const int64_t want = (p.M + rows_per_cta - 1) / rows_per_cta;
  const int64_t cap = int64_t(dev.sm_count) * occ;
  const int grid = int(want < cap ? want : cap);
  WarpArgs a{static_cast<const unsigned char*>(p.x), static_cast<unsigned char*>(p.y), p.m_out, p.d_out,
             p.lse_out, p.M, p.N, uint32_t(p.N * elem_bytes(p.dtype)), plan.slot_bytes, plan.slots, dev.status,
             local_wait_limit_ns()};
  fn<<<grid, threads, plan.smem, p.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace rwo
