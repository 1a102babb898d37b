// kernel_oneread_tma.cu -- one-read softmax with rows staged in shared memory by bulk copies.
//
// "5.2 CUDA Online Softmax 实现优化", §6 keeps the row on chip so that x is read from HBM once
// and y written once; "Softmax 数值稳定性与 IO-Aware Attention" §三 names shared memory as the
// place for rows that fit.  On sm_103a the copy engine does the loading:
//
//  * One producer warp (one elected lane) per CTA issues cp.async.bulk global -> shared for
//    whole rows into a ring of S row slots, completion counted in bytes on an mbarrier per
//    slot ("full").
//  * NCW consumer warps wait on "full", copy their part of the row (VPT 16-byte vectors per
//    thread) into registers and at once hand the slot back ("freed"), so all S slots carry HBM
//    reads in flight while rows are being normalised.  Each thread folds its values into its
//    (m, d) state with one exponential per element, states are merged across the warp
//    (butterfly) and across the consumer warps (shared memory, one named barrier per row), and
//    y = e * 2^((m_t - m) log2 e) / d leaves the registers in 16-byte streaming stores.
//
// Persistent: the grid is (CTAs resident per SM) x (SM count); CTA b handles rows b, b + grid,
// ...  Every wait is bounded (%globaltimer); a wait that runs out sets the status word and the
// protocol continues, so the kernel always terminates.
#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

struct TmaArgs {
  const unsigned char* x;
  unsigned char* y;
  float* m_out;
  float* d_out;
  float* lse_out;
  int64_t M;
  int64_t N;
  uint32_t row_bytes;
  uint32_t slot_bytes;
  int stages;
  unsigned* status;
  uint64_t wait_ns;
  const int64_t* labels;  // state-only mode: cross-entropy labels, or null
  float* loss;
  int64_t x_pitch, y_pitch;  // bytes between rows
  float scale;               // softmax of scale * x
  float c;                   // scale * log2 e
};
// Each copy moves at most slot_bytes: the whole row (slot_bytes >= row_bytes), or in the
// state-only mode, for rows longer than a slot, chunks of slot_bytes (a multiple of 128) and a
// shorter last one -- ceil(row_bytes / slot_bytes) copies per row.

constexpr int kSlotAlign = 128;

// What the kernel writes besides the row state: y = softmax, y = log softmax, or nothing (the
// row state alone, optionally the cross-entropy loss).
enum TmaOut { kTmaProb = 0, kTmaLog = 1, kTmaState = 2 };

// PK (16-bit types, rows of 64 - 128 KiB): the consumers keep x as the packed 16-byte vectors (4
// registers each instead of 8) and form y from them after the merge, a second exponential per
// element in the softmax.
template <class D, int VPT, int NCW, int OUT, bool PK = false>
__global__ void __launch_bounds__((NCW + 1) * 32) k_oneread_tma(TmaArgs a) {
  constexpr bool LOG = OUT == kTmaLog;
  constexpr bool WRITE_Y = OUT != kTmaState;
  static_assert(!PK || WRITE_Y, "the state-only mode packs anyway");
  extern __shared__ __align__(128) unsigned char smem[];
  constexpr int E = D::kVec;
  constexpr int NCT = NCW * 32;
  const int S = a.stages;
  unsigned char* slots = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(S) * a.slot_bytes);
  uint64_t* freed = full + S;
  State* wstate = reinterpret_cast<State*>(freed + S);  // [2][NCW]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&full[s]), 1);
      mbar_init(smem_addr(&freed[s]), NCW);
    }
    fence_mbar_init();
  }
  __syncthreads();

  const int64_t nrows = a.M > blockIdx.x ? (a.M - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  const int64_t nunits = a.N / E;

  if (warp == NCW) {
    // ---------------- producer: keep S row loads in flight ----------------
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      bool timed_out = false;
      int s = 0;         // slot of copy j and the parity of its lap, kept incrementally (a 64-bit
      uint32_t ph = 0;   // division per row would cost ~0.1 us of this lane's time)
      int64_t r = 0;     // this CTA's row and the chunk of it that copy j carries
      int ch = 0;
      // one copy per row where y is written (the row fits a slot); the state-only mode may chunk
      const int nch = WRITE_Y ? 1 : int((a.row_bytes + a.slot_bytes - 1) / a.slot_bytes);
      const int64_t ncopies = nrows * nch;
      for (int64_t j = 0; j < ncopies; ++j) {
        if (j >= S && !mbar_wait(smem_addr(&freed[s]), ph ^ 1u, a.wait_ns)) timed_out = true;
        const uint32_t bar = smem_addr(&full[s]);
        if constexpr (WRITE_Y) {
          mbar_arrive_expect_tx(bar, a.row_bytes);
          const int64_t row = blockIdx.x + j * gridDim.x;
          bulk_g2s(smem_addr(slots + size_t(s) * a.slot_bytes), a.x + row * a.x_pitch, a.row_bytes, bar, pol);
        } else {
          const uint32_t off = uint32_t(ch) * a.slot_bytes;
          const uint32_t bytes = a.row_bytes - off < a.slot_bytes ? a.row_bytes - off : a.slot_bytes;
          mbar_arrive_expect_tx(bar, bytes);
          const int64_t row = blockIdx.x + r * gridDim.x;
          bulk_g2s(smem_addr(slots + size_t(s) * a.slot_bytes), a.x + row * a.x_pitch + off, bytes, bar, pol);
          if (++ch == nch) {
            ch = 0;
            ++r;
          }
        }
        if (++s == S) {
          s = 0;
          ph ^= 1u;
        }
      }
      // Every load must have landed before the CTA may exit (the consumers normally saw them all).
      for (int64_t j = ncopies > S ? ncopies - S : 0; j < ncopies; ++j)
        if (!mbar_wait(smem_addr(&full[j % S]), uint32_t((j / S) & 1), a.wait_ns)) timed_out = true;
      if (timed_out) atomicOr(a.status, kStatusTimeout);
    }
    return;
  }

  // ---------------- consumers ----------------
  bool timed_out = false;
  int cs = 0;  // slot of the next copy and the parity of its lap (state-only mode)
  uint32_t cph = 0;
  for (int64_t j = 0; j < nrows; ++j) {
    // Kept incrementally in the state-only mode, whose consumers set the pace (measured 7% faster
    // on 64 KiB rows); the modes that write y measured 3% faster with the division here.
    int s = 0;
    uint32_t par = 0;
    if constexpr (WRITE_Y) {
      s = int(j % S);
      par = uint32_t((j / S) & 1);
    }
    // cross entropy: thread 0 fetches the label before the row arrives
    int64_t label = -1;
    if constexpr (OUT == kTmaState) {
      if (a.loss && tid == 0) label = a.labels[blockIdx.x + j * gridDim.x];
    }
    uint32_t slot = 0;
    if constexpr (WRITE_Y) {
      if (!mbar_wait(smem_addr(&full[s]), par, a.wait_ns)) timed_out = true;
      slot = smem_addr(slots + size_t(s) * a.slot_bytes);
    }
    float x_label = 0.f;  // the labelled entry, read from the staged row before the slot is freed

    // copy this thread's part of the row into registers and hand the slot back at once
    float mt = -INFINITY, dt = 0.f;
    float v[WRITE_Y && !PK ? VPT : 1][E];  // values kept for the normalisation (unpacked modes)
    uint4 qk[PK ? VPT : 1];                // the same, packed
    if constexpr (PK) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int u = tid + k * NCT;
        qk[k] = u < nunits ? lds16(slot + uint32_t(u) * 16u)
                           : make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&freed[s]));
      mt = D::vmax_all(qk);
      const float mts = safe_max(mt);
      const float2 nms = make_float2(-mts, -mts);
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        float2 f[E / 2];
        D::unpack2(qk[k], f);
#pragma unroll
        for (int e = 0; e < E / 2; ++e) acc = __fadd2_rn(acc, exp_diff2(f[e], nms, a.c));
      }
      dt = __fadd_rn(acc.x, acc.y);
    } else if constexpr (WRITE_Y) {
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int u = tid + k * NCT;
        if (u < nunits) {
          D::unpack(lds16(slot + uint32_t(u) * 16u), v[k]);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) v[k][e] = -INFINITY;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&freed[s]));

#pragma unroll
      for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) mt = fmaxf(mt, v[k][e]);
      const float mts = safe_max(mt);
#pragma unroll
      for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if constexpr (LOG) {  // x stays in registers for y = scale (x - m) - ln d
            dt += exp_diff(v[k][e], mts, a.c);
          } else {
            v[k][e] = exp_diff(v[k][e], mts, a.c);
            dt += v[k][e];
          }
        }
    } else {
      // State only: the row arrives in nch chunks (one unless it is longer than a slot), each
      // folded into the thread's running state with the (m, d) merge.  Per chunk: keep the packed
      // vectors, take the max on them (packed bf16 max), then the exponentials in pairs (packed
      // f32x2 add and multiply).  For one chunk the merge with the empty state returns the
      // chunk's state bit for bit.  Slots are counted incrementally here (measured 7% faster on
      // 64 KiB rows than the division the other modes use).
      const int64_t chunk_units = int64_t(a.slot_bytes) / 16;
      const int nch = int((a.row_bytes + a.slot_bytes - 1) / a.slot_bytes);
      State run = empty_state();
      for (int ch = 0; ch < nch; ++ch) {
        s = cs;
        par = cph;
        if (++cs == S) {
          cs = 0;
          cph ^= 1u;
        }
        if (!mbar_wait(smem_addr(&full[s]), par, a.wait_ns)) timed_out = true;
        slot = smem_addr(slots + size_t(s) * a.slot_bytes);
        const int64_t u0 = int64_t(ch) * chunk_units;  // the chunk's first unit in the row
        const int64_t cu = nunits - u0 < chunk_units ? nunits - u0 : chunk_units;
        if (a.loss && tid == 0 && label >= u0 * E && label < (u0 + cu) * E)
          x_label = D::lds1(slot, label - u0 * E);
        uint4 q[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
          const int u = tid + k * NCT;
          q[k] = u < cu ? lds16(slot + uint32_t(u) * 16u)
                        : make_uint4(D::kNegInfWord, D::kNegInfWord, D::kNegInfWord, D::kNegInfWord);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&freed[s]));
        const float mc = D::vmax_all(q);
        const float mcs = safe_max(mc);
        float2 acc = make_float2(0.f, 0.f);
        float dc;
        if (exp_shift_ok(mcs)) {
          const ExpShift sh = exp_shift(mcs, a.c);
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            float2 f[E / 2];
            D::unpack2(q[k], f);
#pragma unroll
            for (int e = 0; e < E / 2; ++e) acc = __fadd2_rn(acc, exp_shifted2(f[e], sh));
          }
          dc = __fmul_rn(__fadd_rn(acc.x, acc.y), sh.unscale);
        } else {
          const float2 nms = make_float2(-mcs, -mcs);
#pragma unroll
          for (int k = 0; k < VPT; ++k) {
            float2 f[E / 2];
            D::unpack2(q[k], f);
#pragma unroll
            for (int e = 0; e < E / 2; ++e) acc = __fadd2_rn(acc, exp_diff2(f[e], nms, a.c));
          }
          dc = __fadd_rn(acc.x, acc.y);
        }
        run = merge(run, State{mc, dc}, a.c);
      }
      mt = run.m;
      dt = run.d;
    }
    State st;
    if constexpr (WRITE_Y)
      st = group_merge(
          State{mt, dt}, wstate + (j & 1) * NCW, NCW, warp, lane, [] { named_barrier_sync(1, NCT); }, a.c);
    else
      st = group_merge_nary(
          State{mt, dt}, wstate + (j & 1) * NCW, NCW, warp, lane, [] { named_barrier_sync(1, NCT); }, a.c);
    const int64_t row = blockIdx.x + j * gridDim.x;
    if constexpr (PK) {
      // y from the packed x: softmax 2^((x - m) c) / d, log softmax (x - m) scale - ln d, in pairs
      unsigned char* yr = a.y + row * a.y_pitch;
      const LogNorm ln = log_norm(st);
      const float ms = safe_max(st.m);
      const float2 nms = make_float2(-ms, -ms), inv2 = make_float2(safe_inv(st.d), safe_inv(st.d));
      const float2 sc2 = make_float2(a.scale, a.scale), nlnd2 = make_float2(-ln.lnd, -ln.lnd);
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int u = tid + k * NCT;
        if (u < nunits) {
          float2 f[E / 2];
          D::unpack2(qk[k], f);
#pragma unroll
          for (int e = 0; e < E / 2; ++e)
            f[e] = LOG ? __ffma2_rn(__fadd2_rn(f[e], nms), sc2, nlnd2) : __fmul2_rn(exp_diff2(f[e], nms, a.c), inv2);
          st_stream16(yr + int64_t(u) * 16, D::pack2(f));
        }
      }
    } else if constexpr (WRITE_Y) {
      float scale = 0.f;
      LogNorm ln{};
      if constexpr (LOG) ln = log_norm(st);
      else scale = __fmul_rn(exp_diff(mt, safe_max(st.m), a.c), safe_inv(st.d));
      unsigned char* yr = a.y + row * a.y_pitch;
#pragma unroll
      for (int k = 0; k < VPT; ++k) {
        const int u = tid + k * NCT;
        if (u < nunits) {
#pragma unroll
          for (int e = 0; e < E; ++e) v[k][e] = LOG ? log_prob(v[k][e], ln, a.scale) : __fmul_rn(v[k][e], scale);
          st_stream16(yr + int64_t(u) * 16, D::pack(v[k]));
        }
      }
    }
    if (tid == 0) {
      const State o = scaled_state(st, a.scale);
      if (a.m_out) a.m_out[row] = o.m;
      if (a.d_out) a.d_out[row] = o.d;
      if (a.lse_out) a.lse_out[row] = lse_of(o);
      if constexpr (OUT == kTmaState) {
        // cross entropy ("从原始Softmax到在线Softmax", "交叉熵损失计算"); negative label: ignored
        // row (0); label >= N: NaN and a status bit, x not read
        if (a.loss) {
          float l = 0.f;
          if (label >= a.N) {
            l = __int_as_float(0x7fc00000);
            atomicOr(a.status, kStatusBadLabel);
          } else if (label >= 0) {
            l = ce_loss(st, x_label, a.scale);
          }
          a.loss[row] = l;
        }
      }
    }
  }
  if (timed_out && lane == 0) atomicOr(a.status, kStatusTimeout);
}

using TmaKernel = void (*)(TmaArgs);

struct TmaConfig {
  int ncw, vpt;
  TmaKernel fn[3][3];  // [output mode][dtype]
};

template <int VPT, int NCW>
constexpr TmaConfig tma_cfg() {
  return TmaConfig{NCW, VPT,
                   {{k_oneread_tma<F32, VPT, NCW, kTmaProb>, k_oneread_tma<BF16, VPT, NCW, kTmaProb>,
                     k_oneread_tma<F16, VPT, NCW, kTmaProb>},
                    {k_oneread_tma<F32, VPT, NCW, kTmaLog>, k_oneread_tma<BF16, VPT, NCW, kTmaLog>,
                     k_oneread_tma<F16, VPT, NCW, kTmaLog>},
                    {k_oneread_tma<F32, VPT, NCW, kTmaState>, k_oneread_tma<BF16, VPT, NCW, kTmaState>,
                     k_oneread_tma<F16, VPT, NCW, kTmaState>}}};
}

// fp32 rows of 64 - 128 KiB: 10, 12 or 16 vectors a thread over 16 warps (one CTA per SM).
// 16-bit rows of 64 - 120 KiB: the vectors kept packed, 10, 12, 14 or 16 a thread over 15 warps
// (16 warps in all, so that a thread may take 128 registers: with 17 warps on four sub-partitions
// it gets 96, and even the packed form spilled; 14 and 16 vectors still spill 28-96 bytes and
// measured 6.3-6.5 TB/s all the same, bf16 112 / 120 KiB 6.32 / 6.38 against 5.13 / 5.30 on two
// passes).  The state-only mode streams such rows in chunks
// through the smaller configurations and has no entry here.
template <int VPT>
constexpr TmaConfig tma_cfg_wide() {
  return TmaConfig{16, VPT,
                   {{k_oneread_tma<F32, VPT, 16, kTmaProb>, nullptr, nullptr},
                    {k_oneread_tma<F32, VPT, 16, kTmaLog>, nullptr, nullptr},
                    {nullptr, nullptr, nullptr}}};
}
template <int VPT>
constexpr TmaConfig tma_cfg_packed() {
  return TmaConfig{15, VPT,
                   {{nullptr, k_oneread_tma<BF16, VPT, 15, kTmaProb, true>, k_oneread_tma<F16, VPT, 15, kTmaProb, true>},
                    {nullptr, k_oneread_tma<BF16, VPT, 15, kTmaLog, true>, k_oneread_tma<F16, VPT, 15, kTmaLog, true>},
                    {nullptr, nullptr, nullptr}}};
}
const TmaConfig kTmaPacked[] = {tma_cfg_packed<10>(), tma_cfg_packed<12>(), tma_cfg_packed<14>(), tma_cfg_packed<16>()};
template <int VPT, int NCW>
constexpr TmaConfig tma_cfg_packed_n() {  // 16-bit types, x kept packed
  return TmaConfig{NCW, VPT,
                   {{nullptr, k_oneread_tma<BF16, VPT, NCW, kTmaProb, true>, k_oneread_tma<F16, VPT, NCW, kTmaProb, true>},
                    {nullptr, k_oneread_tma<BF16, VPT, NCW, kTmaLog, true>, k_oneread_tma<F16, VPT, NCW, kTmaLog, true>},
                    {nullptr, nullptr, nullptr}}};
}
// 16-bit rows of 32 - 54 KiB: packed too, 8, 10, 12 or 14 vectors a thread over 8 consumer warps
// (measured, bf16, ~1 GB per launch, softmax / log softmax TB/s against the unpacked
// configurations: 32 KiB 6.08 / 6.14 against 6.04 / 5.65, 36 KiB 6.38 / 6.73 against 5.01 /
// 4.69, 40 KiB 6.81 against 5.34, 44 KiB 6.61 / 6.73 against 5.74 / 5.39, 48 KiB 6.89 against
// 6.01, 52 KiB 6.82 / 6.37 against 6.37 / 6.00, 54 KiB 6.55 / 6.29 against 6.50 / 6.16; but
// 24 KiB 6.18 against 6.33, 56 KiB 6.43 against 6.53, 64 KiB 6.16 against 6.86).
// 16-bit rows of 8 - 16 KiB: packed, 8 vectors a thread over 4 consumer warps, with the CTAs per
// SM chosen so that about 84 KiB of rows are in flight per SM (plan_tma) -- more measured slower.
// bf16, ~1 GB per launch, TB/s at 2 / 3 / 4 CTAs per SM: 10 KiB 4.72 / 5.64 / 6.17, 12 KiB 5.48 /
// 6.50 / 6.05, 14 KiB 6.17 / 6.29 / 5.91, 16 KiB 6.63 / 6.04 / 5.99, against 4.87 / 5.67 / 6.22 /
// 5.98 for the unpacked configurations and 5.32 (12 KiB) / 5.48 (16 KiB) for the register kernel.
const TmaConfig kTmaPacked4 = tma_cfg_packed_n<8, 4>();
constexpr int64_t kPacked4InFlight = 86016;

// fp32 rows of 8 - 16 KiB where y is written: 8 vectors a thread over 4 consumer warps, at most 4
// CTAs per SM (measured on fp32 4096 x 4096: 22.60 against 23.26 us for 4 vectors over 8 warps;
// 5 - 8 CTAs per SM 22.65 - 22.85).  Only forced or pitched rows reach it: AUTO keeps fp32 rows up
// to 64 KiB in registers.
const TmaConfig kTmaF32Short = tma_cfg<8, 4>();
constexpr int kF32ShortCtas = 4;

const TmaConfig kTmaPacked8[] = {tma_cfg_packed_n<8, 8>(), tma_cfg_packed_n<10, 8>(), tma_cfg_packed_n<12, 8>(),
                                 tma_cfg_packed_n<14, 8>()};

// Ordered by capacity (16-byte units per row = 32 * ncw * vpt).
const TmaConfig kTma[] = {tma_cfg<2, 4>(),          tma_cfg<4, 4>(),          tma_cfg<4, 8>(),
                          tma_cfg<8, 8>(),          tma_cfg<8, 16>(),         tma_cfg_wide<10>(),
                          tma_cfg_wide<12>(),   tma_cfg_wide<16>()};
constexpr int kTmaWide16 = 7;  // index of the 16-vector fp32 configuration

// The smallest configuration that holds the row, except fp32 rows of 8 - 16 KiB (4 consumer warps)
// and of 64 - 68 KiB, which take the 16-vector one (with two slots: see plan_tma), and 16-bit rows of 32 - 54 KiB and above 64 KiB,
// kept packed, and 16-bit rows of 8 - 16 KiB (packed over 4 consumer warps).  The state-only mode
// (which keeps x packed anyway, and sees at most 32 KiB at a time) takes the plain configurations.
const TmaConfig* pick_tma(int64_t units, int dtype, bool state) {
  if (dtype == 0 && !state && units > 512 && units <= 1024) return &kTmaF32Short;
  if (dtype == 0 && !state && units > 4096 && units <= 4352) return &kTma[kTmaWide16];  // fp32
  if (dtype != 0 && !state && units > 512 && units <= 1024) return &kTmaPacked4;  // 16-bit, 8 - 16 KiB
  if (dtype != 0 && !state && units >= 2048 && units <= 3456) {  // 16-bit rows of 32 - 54 KiB
    for (const TmaConfig& c : kTmaPacked8)
      if (units <= int64_t(32) * c.ncw * c.vpt) return &c;
  }
  if (dtype != 0 && !state && units > 4096) {
    for (const TmaConfig& c : kTmaPacked)
      if (units <= int64_t(32) * c.ncw * c.vpt) return &c;
    return nullptr;
  }
  for (const TmaConfig& c : kTma)
    if (units <= int64_t(32) * c.ncw * c.vpt) return c.fn[0][dtype] ? &c : nullptr;
  return nullptr;
}

struct TmaPlan {
  const TmaConfig* cfg = nullptr;
  int stages = 0;
  uint32_t slot_bytes = 0;
  size_t smem = 0;
  int ctas_per_sm = 0;
};

size_t tma_smem_bytes(int stages, uint32_t slot_bytes, int ncw) {
  return size_t(stages) * slot_bytes + size_t(stages) * 2 * sizeof(uint64_t) +
         size_t(2) * ncw * sizeof(State);
}

// Two row slots per CTA, then as many CTAs per SM as shared memory and threads allow (measured
// against 4 slots for rows up to 16 KiB and 3 above: fp32 4096 x 4096 24.1 -> 22.9 us, fp32 48 KiB
// rows 336 -> 325 us, 64 KiB 360 -> 358 us, bf16 64 KiB rows unchanged).  fp32 rows above 68 KiB
// take one slot: the consumers free it as soon as the row is in registers, so the next row's load
// still overlaps this row's normalisation and stores (measured, 8000 rows, TB/s one slot / two:
// 16 vectors a thread 64 KiB 5.62 / 6.58, 68 KiB 5.77 / 6.43, 80 KiB 6.10 / 5.83, 112 KiB 6.68 /
// 5.93; the fitted 10 and 12 vectors with one slot 72 KiB 6.28, 80 KiB 6.47, 88 KiB 6.56, 96 KiB
// 6.68; 128 KiB (one slot only) 6.38).  16-bit rows of 64 - 120 KiB, x kept packed (bf16, ~1 GB
// per launch, softmax / log softmax TB/s, one slot against two): 64 KiB + 16 B 5.96 / 5.82
// against 6.28 / 6.50, 80 KiB 6.20 / 5.98 against 6.18 / 6.25, 88 KiB 6.44 / 6.24 against
// 6.20 / 6.15, 98 KiB 6.30 / 6.36 against 5.85 / 6.10, 105 KiB 6.43 / 6.48 against 6.09 / 6.20
// (two passes: 4.66-5.02).
// The state-only mode (row state, cross entropy) needs each element once and nothing kept, so rows
// longer than 32 KiB stream through the slots in 32 KiB chunks, any length: measured (bf16,
// ~1 GB per launch, cross entropy) 6.7-7.1 TB/s for rows of 64 - 297 KiB against 2.8-5.0 on the
// two-pass kernel's first pass, and 6.7 against 6.3 TB/s for 64 KiB rows copied whole; 64 KiB
// chunks measured 4.8-7.1.
constexpr int64_t kStateChunk = 32768;

TmaPlan plan_tma(const RowProblem& p, const DeviceInfo& dev) {
  TmaPlan plan;
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  if (row_bytes % 16 != 0) return plan;
  int64_t copy_bytes = row_bytes;
  const TmaConfig* cfg = nullptr;
  if (p.y == nullptr && row_bytes > kStateChunk) {
    // state only: the row streams through the slots in chunks (rows below 4 GiB)
    if (row_bytes >= (int64_t(1) << 32)) return plan;
    copy_bytes = kStateChunk;
    cfg = pick_tma(kStateChunk / 16, p.dtype, true);
  } else {
    if (row_bytes > (int64_t(1) << 20)) return plan;
    cfg = pick_tma(row_bytes / 16, p.dtype, p.y == nullptr);
  }
  if (!cfg) return plan;
  const uint32_t slot = uint32_t((copy_bytes + kSlotAlign - 1) / kSlotAlign * kSlotAlign);
  const size_t per_cta_reserved = 1024;  // the runtime's per-block reservation
  const int threads = (cfg->ncw + 1) * 32;
  // one slot for fp32 rows above 68 KiB and 16-bit rows above 80 KiB, and for 16-bit rows of 32 KiB
  // on the packed 8-warp configuration, which fits two CTAs per SM (bf16, ~1 GB per launch:
  // softmax / log softmax 6.61 / 6.57 TB/s against 6.01 / 6.12 with two slots; from 34 KiB on,
  // one CTA per SM, one slot measured 5.1 - 5.9 against 6.2 - 6.9)
  const int first = copy_bytes > (p.dtype == 0 ? 69632 : 81920) || cfg == &kTmaPacked8[0] ? 1 : 2;
  for (int stages = first; stages >= 1; --stages) {
    const size_t smem = tma_smem_bytes(stages, slot, cfg->ncw);
    if (smem > size_t(dev.max_smem_per_block_optin)) continue;
    int by_smem = int(size_t(dev.max_smem_per_sm) / (smem + per_cta_reserved));
    int by_threads = dev.max_threads_per_sm / threads;
    int c = by_smem < by_threads ? by_smem : by_threads;
    if (c > 8) c = 8;
    if (cfg == &kTmaF32Short && c > kF32ShortCtas) c = kF32ShortCtas;
    if (cfg == &kTmaPacked4) {  // about kPacked4InFlight bytes of rows in flight per SM, 2 - 4 CTAs
      const int64_t want = kPacked4InFlight / (int64_t(stages) * int64_t(slot));
      const int w = want < 2 ? 2 : want > 4 ? 4 : int(want);
      if (c > w) c = w;
    }
    if (c < 1) continue;
    plan.cfg = cfg;
    plan.stages = stages;
    plan.slot_bytes = slot;
    plan.smem = smem;
    plan.ctas_per_sm = c;
    return plan;
  }
  return plan;
}

}  // namespace

bool oneread_tma_fits(const RowProblem& p, const DeviceInfo& dev) {
  return plan_tma(p, dev).cfg != nullptr;
}

cudaError_t launch_oneread_tma(const RowProblem& p, const DeviceInfo& dev) {
  const TmaPlan plan = plan_tma(p, dev);
  if (!plan.cfg) return cudaErrorInvalidValue;
  const int out = p.y == nullptr ? kTmaState : p.log_out ? kTmaLog : kTmaProb;
  if (p.loss && out != kTmaState) return cudaErrorInvalidValue;
  TmaKernel fn = plan.cfg->fn[out][p.dtype];
  if (!fn) return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute((const void*)fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(plan.smem));
  if (err != cudaSuccess) return err;
  const int threads = (plan.cfg->ncw + 1) * 32;
  int occ = 0;
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, (const void*)fn, threads, plan.smem);
  if (err != cudaSuccess) return err;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  int per_sm = plan.ctas_per_sm < occ ? plan.ctas_per_sm : occ;
  const int64_t cap = int64_t(dev.sm_count) * per_sm;
  const int grid = int(p.M < cap ? p.M : cap);
  TmaArgs a{static_cast<const unsigned char*>(p.x), static_cast<unsigned char*>(p.y), p.m_out,
            p.d_out, p.lse_out, p.M, p.N, uint32_t(p.N * elem_bytes(p.dtype)), plan.slot_bytes,
            plan.stages, dev.status, local_wait_limit_ns(), p.labels, p.loss,
            p.x_pitch ? p.x_pitch : int64_t(p.N) * elem_bytes(p.dtype),
            p.y_pitch ? p.y_pitch : int64_t(p.N) * elem_bytes(p.dtype), p.scale, p.scale * kLog2e};
  fn<<<grid, threads, plan.smem, p.stream>>>(a);
  return cudaGetLastError();
}

}  // namespace rwo
