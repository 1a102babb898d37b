// kernels_rowwise.cu -- register one-read kernel, two-pass streaming kernel, state merge kernel.
//
// Register one-read ("5.2 CUDA Online Softmax 实现优化", §6: keep the row on chip so x is
// read once and y written once).  A group of WPR warps owns a row; each thread loads VPT
// 16-byte vectors (or VPT scalars on the unaligned path) into registers, takes its local
// max, forms e = 2^((x - m_t) log2 e) once per element and sums it: the thread's (m, d)
// state.  States are merged across the warp by a butterfly and across the group's warps
// through shared memory; then y = e * 2^((m_t - m) log2 e) / d is stored from the same
// registers.  One exponential per element.  Up to kGridWaves waves of CTAs take one row group
// each; beyond that, CTAs walk rows with a grid stride (§7 of the same page).
//
// Two-pass ("5.2 ..." §2.2 and §5: the online recurrence with 128-bit loads).  A CTA owns a
// row.  Pass 1 streams the row, four vectors per thread per step, folding each step into
// the thread's (m, d) with one rescale (the online recurrence at step granularity) and a
// compensated sum; the block merge gives the row state; pass 2 re-reads the row (from L2
// while it is resident) and writes y.  Any N.  With WRITE_Y = false it is the state-only
// kernel behind softmax_row_state.
//
// Merge kernel: the elementwise state merge ("5.2 ..." §4.1) behind merge_states.
#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

struct RowArgs {
  const unsigned char* x;
  unsigned char* y;
  float* m_out;
  float* d_out;
  float* lse_out;
  int64_t M;
  int64_t N;
  int64_t q_period;    // causal rule (two-pass causal mode only): row r keeps its first
  int64_t key_offset;  // clamp(r % q_period + 1 + key_offset, 0, N) entries
  const int64_t* labels;  // cross entropy (two-pass state mode only), else null
  float* loss;
  unsigned* status;
  int64_t x_pitch, y_pitch;  // bytes between rows
  float scale;               // softmax of scale * x
  float c;                   // scale * log2 e: the exponent slope
};

// Row outputs for the softmax of scale * x (s holds the raw maximum).
__device__ __forceinline__ void write_state(const RowArgs& a, int64_t row, State s) {
  const State o = scaled_state(s, a.scale);
  if (a.m_out) a.m_out[row] = o.m;
  if (a.d_out) a.d_out[row] = o.d;
  if (a.lse_out) a.lse_out[row] = lse_of(o);
}

// Cross entropy of row `row` against its label ("从原始Softmax到在线Softmax", section
// "交叉熵损失计算": loss = -log p_label).  A negative label marks a row to
// ignore (loss 0); a label >= N gives NaN and sets kStatusBadLabel, without reading x there.
template <class D>
__device__ __forceinline__ void write_loss(const RowArgs& a, int64_t row, const unsigned char* xr, State s) {
  const int64_t label = a.labels[row];
  float l;
  if (label < 0) {
    l = 0.f;
  } else if (label >= a.N) {
    l = __int_as_float(0x7fc00000);
    atomicOr(a.status, kStatusBadLabel);
  } else {
    l = ce_loss(s, D::load1(xr, label), a.scale);
  }
  a.loss[row] = l;
}

// ------------------------------------------------------------------------------------------
// Register one-read kernel
// ------------------------------------------------------------------------------------------

constexpr int kRegThreads = 256;
constexpr int kGridWaves = 8;  // CTAs launched per resident CTA slot before rows are walked

template <class D, int VPT, int WPR, bool VEC, bool LOG>
__global__ void __launch_bounds__(kRegThreads) k_oneread_reg(RowArgs a) {
  constexpr int E = VEC ? D::kVec : 1;  // elements per unit (one 16-byte vector, or one element)
  constexpr int G = (kRegThreads / 32) / WPR;  // row groups per CTA
  constexpr int GT = WPR * 32;                 // threads per group
  __shared__ State slots[2][kRegThreads / 32];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = warp / WPR, wig = warp % WPR;
  const int gt = threadIdx.x - g * GT;
  const int64_t nunits = a.N / E;

  int it = 0;
  for (int64_t row = (int64_t)blockIdx.x * G + g; row < a.M; row += (int64_t)gridDim.x * G, ++it) {
    const unsigned char* xr = a.x + row * a.x_pitch;
    float v[VPT][E];
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t u = gt + (int64_t)k * GT;
      if (u < nunits) {
        if constexpr (VEC) {
          D::unpack(ld_stream16(xr + u * 16), v[k]);
        } else {
          v[k][0] = D::load1(xr, u);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) v[k][e] = -INFINITY;
      }
    }
    // thread state: local max first, then one exponential per element
    float mt = -INFINITY;
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
      for (int e = 0; e < E; ++e) mt = fmaxf(mt, v[k][e]);
    const float mts = safe_max(mt);
    float dt = 0.f;
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
    const State s = group_merge(
        State{mt, dt}, &slots[it & 1][g * WPR], WPR, wig, lane, [&] { named_barrier_sync(1 + g, GT); }, a.c);
    float scale = 0.f;
    LogNorm ln{};
    if constexpr (LOG) ln = log_norm(s);
    else scale = __fmul_rn(exp_diff(mt, safe_max(s.m), a.c), safe_inv(s.d));
    unsigned char* yr = a.y + row * a.y_pitch;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
      const int64_t u = gt + (int64_t)k * GT;
      if (u < nunits) {
#pragma unroll
        for (int e = 0; e < E; ++e) v[k][e] = LOG ? log_prob(v[k][e], ln, a.scale) : __fmul_rn(v[k][e], scale);
        if constexpr (VEC) {
          st_stream16(yr + u * 16, D::pack(v[k]));
        } else {
          D::store1(yr, u, v[k][0]);
        }
      }
    }
    if (gt == 0) write_state(a, row, s);
  }
}

using RowKernel = void (*)(RowArgs);

struct RegConfig {
  int wpr, vpt;
  RowKernel fn[2][3];  // [log output][dtype]
};

template <int VPT, int WPR, bool VEC>
constexpr RegConfig reg_cfg() {
  return RegConfig{WPR, VPT,
                   {{k_oneread_reg<F32, VPT, WPR, VEC, false>, k_oneread_reg<BF16, VPT, WPR, VEC, false>,
                     k_oneread_reg<F16, VPT, WPR, VEC, false>},
                    {k_oneread_reg<F32, VPT, WPR, VEC, true>, k_oneread_reg<BF16, VPT, WPR, VEC, true>,
                     k_oneread_reg<F16, VPT, WPR, VEC, true>}}};
}

// Ordered by capacity (units per row = 32 * wpr * vpt).
const RegConfig kRegVec[] = {reg_cfg<2, 1, true>(), reg_cfg<4, 1, true>(), reg_cfg<8, 1, true>(),
                             reg_cfg<8, 2, true>(), reg_cfg<8, 4, true>(), reg_cfg<8, 8, true>(),
                             reg_cfg<12, 8, true>(), reg_cfg<16, 8, true>()};
const RegConfig kRegScalar[] = {reg_cfg<4, 1, false>(), reg_cfg<16, 1, false>(),
                                reg_cfg<8, 8, false>()};

// 16-bit rows of 3 - 4 KiB: 4 vectors a thread over two warps per row instead of 8 over one (bf16
// and fp16 4 KiB rows, ~1 GB per launch: 6.75 against 6.22 TB/s; 3 KiB 6.02 against 6.00; fp32
// rows of the same units already hold half the values a thread).
const RegConfig kReg16Mid = reg_cfg<4, 2, true>();

const RegConfig* pick_reg(int64_t units, bool vec, int dtype) {
  if (vec && dtype != 0 && units > 192 && units <= 256) return &kReg16Mid;
  const RegConfig* tab = vec ? kRegVec : kRegScalar;
  const int n = vec ? int(sizeof(kRegVec) / sizeof(kRegVec[0]))
                    : int(sizeof(kRegScalar) / sizeof(kRegScalar[0]));
  for (int i = 0; i < n; ++i)
    if (units <= int64_t(32) * tab[i].wpr * tab[i].vpt) return &tab[i];
  return nullptr;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int blocks_per_sm(const void* fn, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, threads, smem) != cudaSuccess) {
    cudaGetLastError();
    n = 1;
  }
  return n < 1 ? 1 : n;
}

RowArgs row_args(const RowProblem& p, const DeviceInfo& dev) {
  const int64_t row_bytes = p.N * elem_bytes(p.dtype);
  return RowArgs{static_cast<const unsigned char*>(p.x), static_cast<unsigned char*>(p.y),
                 p.m_out, p.d_out, p.lse_out, p.M, p.N, 1, 0, p.labels, p.loss, dev.status,
                 p.x_pitch ? p.x_pitch : row_bytes, p.y_pitch ? p.y_pitch : row_bytes, p.scale,
                 p.scale * kLog2e};
}

// ------------------------------------------------------------------------------------------
// Two-pass streaming kernel
// ------------------------------------------------------------------------------------------

constexpr int kTwoPassMaxThreads = 1024;
constexpr int kTwoPassUnroll = 4;

template <class D, bool VEC>
__device__ __forceinline__ void load_unit(const unsigned char* xr, int64_t u, int64_t nunits,
                                          float (&v)[VEC ? D::kVec : 1]) {
  constexpr int E = VEC ? D::kVec : 1;
  if (u < nunits) {
    if constexpr (VEC) {
      D::unpack(ld16(xr + u * 16), v);
    } else {
      v[0] = D::load1(xr, u);
    }
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = -INFINITY;
  }
}

// What the two-pass kernel writes.
enum TwoPassMode { kProb = 0, kProbCausal = 1, kLogProb = 2, kStateOnly = 3 };

template <class D, bool VEC, int MODE>
__global__ void __launch_bounds__(kTwoPassMaxThreads) k_twopass(RowArgs a) {
  constexpr bool WRITE_Y = MODE != kStateOnly;
  constexpr bool CAUSAL = MODE == kProbCausal;
  constexpr bool LOG = MODE == kLogProb;
  constexpr int E = VEC ? D::kVec : 1;
  constexpr int U = kTwoPassUnroll;
  __shared__ State slots[2][kTwoPassMaxThreads / 32];
  const int nt = blockDim.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nunits = a.N / E;

  int it = 0;
  for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x, ++it) {
    const unsigned char* xr = a.x + row * a.x_pitch;
    // live elements and units: all of them, or the causal prefix (the rest is never read)
    int64_t L = a.N;
    if constexpr (CAUSAL) {
      L = row % a.q_period + 1 + a.key_offset;
      L = L < 0 ? 0 : (L > a.N ? a.N : L);
    }
    const int64_t lunits = CAUSAL ? (L + E - 1) / E : nunits;
    // pass 1: online fold, one rescale per step of U units; compensated (Kahan) sum of d
    float m = -INFINITY, d = 0.f, c = 0.f;
    for (int64_t base = threadIdx.x; base < lunits; base += (int64_t)nt * U) {
      float v[U][E];
#pragma unroll
      for (int k = 0; k < U; ++k) {
        load_unit<D, VEC>(xr, base + (int64_t)k * nt, lunits, v[k]);
        if constexpr (CAUSAL && E > 1) {  // the vector straddling the live length
          const int64_t keep = L - (base + (int64_t)k * nt) * E;
          if (keep > 0 && keep < E) {
#pragma unroll
            for (int e = 0; e < E; ++e)
              if (e >= keep) v[k][e] = -INFINITY;
          }
        }
      }
      float mu = -INFINITY;
#pragma unroll
      for (int k = 0; k < U; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) mu = fmaxf(mu, v[k][e]);
      const float m_new = fmaxf(m, mu);
      const float ms = safe_max(m_new);
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < U; ++k)
#pragma unroll
        for (int e = 0; e < E; ++e) acc += exp_diff(v[k][e], ms, a.c);
      const float r = exp_diff(m, ms, a.c);  // rescale of the running sum; 0 when m was -inf
      const float ds = __fmul_rn(d, r);
      c = __fmul_rn(c, r);
      const float yk = __fsub_rn(acc, c);
      const float t = __fadd_rn(ds, yk);
      c = __fsub_rn(__fsub_rn(t, ds), yk);
      d = t;
      m = m_new;
    }
    const State s = group_merge(State{m, d}, slots[it & 1], nt >> 5, warp, lane, [] { __syncthreads(); }, a.c);
    if constexpr (WRITE_Y) {
      // pass 2: re-read and normalise
      const float ms = safe_max(s.m);
      const float inv = safe_inv(s.d);
      const LogNorm ln = log_norm(s);
      unsigned char* yr = a.y + row * a.y_pitch;
      for (int64_t base = threadIdx.x; base < nunits; base += (int64_t)nt * U) {
        float v[U][E];
#pragma unroll
        for (int k = 0; k < U; ++k) load_unit<D, VEC>(xr, base + (int64_t)k * nt, lunits, v[k]);
#pragma unroll
        for (int k = 0; k < U; ++k) {
          const int64_t u = base + (int64_t)k * nt;
          if (u < nunits) {
            if constexpr (CAUSAL && E > 1) {  // entries past L count as -inf: y = 0 there
              const int64_t keep = L - u * E;
              if (keep > 0 && keep < E) {
#pragma unroll
                for (int e = 0; e < E; ++e)
                  if (e >= keep) v[k][e] = -INFINITY;
              }
            }
#pragma unroll
            for (int e = 0; e < E; ++e)
              v[k][e] = LOG ? log_prob(v[k][e], ln, a.scale) : __fmul_rn(exp_diff(v[k][e], ms, a.c), inv);
            if constexpr (VEC) {
              st_stream16(yr + u * 16, D::pack(v[k]));
            } else {
              D::store1(yr, u, v[k][0]);
            }
          }
        }
      }
    }
    if (threadIdx.x == 0) {
      write_state(a, row, s);
      if constexpr (MODE == kStateOnly) {
        if (a.loss) write_loss<D>(a, row, xr, s);
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// Elementwise state merge
// ------------------------------------------------------------------------------------------

__global__ void __launch_bounds__(256)
    k_merge_states(const float* __restrict__ m_a, const float* __restrict__ d_a,
                   const float* __restrict__ m_b, const float* __restrict__ d_b, float* m_out,
                   float* d_out, float* lse_out, int64_t M) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < M;
       i += (int64_t)gridDim.x * blockDim.x) {
    const State s = merge(State{m_a[i], d_a[i]}, State{m_b[i], d_b[i]});
    m_out[i] = s.m;
    d_out[i] = s.d;
    if (lse_out) lse_out[i] = lse_of(s);
  }
}

}  // namespace

bool oneread_reg_fits(const RowProblem& p, bool vec) {
  const int64_t e = vec ? 16 / elem_bytes(p.dtype) : 1;
  if (vec && p.N % e != 0) return false;
  return pick_reg(p.N / e, vec, p.dtype) != nullptr;
}

cudaError_t launch_oneread_reg(const RowProblem& p, bool vec, const DeviceInfo& dev) {
  const int64_t e = vec ? 16 / elem_bytes(p.dtype) : 1;
  const RegConfig* cfg = pick_reg(p.N / e, vec, p.dtype);
  if (!cfg) return cudaErrorInvalidValue;
  RowKernel fn = cfg->fn[p.log_out ? 1 : 0][p.dtype];
  const int groups = (kRegThreads / 32) / cfg->wpr;
  const int64_t want = ceil_div(p.M, groups);
  // Up to kGridWaves waves of CTAs, one row group each, before the grid stride takes over: the
  // hardware hands a finished SM the next CTA, which balances SMs that run at different speeds
  // (measured: 4096 x 4096 fp32 21.5 -> 20.9 us, 262144 x 256 fp32 93 -> 80 us against one
  // resident wave walking the rows).
  // Rows in host memory: one resident wave (measured on the host-link path: 254 GB/s against 247
  // with 8 waves, whose extra CTAs only add requests in flight on an already saturated link).
  const int64_t waves = p.host_mem ? 1 : kGridWaves;
  const int64_t cap = int64_t(dev.sm_count) * blocks_per_sm((const void*)fn, kRegThreads, 0) * waves;
  const int grid = int(want < cap ? want : cap);
  fn<<<grid, kRegThreads, 0, p.stream>>>(row_args(p, dev));
  return cudaGetLastError();
}

cudaError_t launch_twopass(const RowProblem& p, bool vec, const DeviceInfo& dev, int64_t q_period,
                           int64_t key_offset) {
  const int64_t e = vec ? 16 / elem_bytes(p.dtype) : 1;
  if (vec && p.N % e != 0) return cudaErrorInvalidValue;
  const int64_t units = p.N / e;
  // Threads per row: from one warp, doubled while a thread would take more than two steps of
  // kTwoPassUnroll vectors (measured: 4096 x 4096 fp32 24.9 -> 22.5 us against one step per
  // thread; 262144 x 256 fp32 358 -> 115 us against a 128-thread minimum).
  int nt = 32;
  while (nt < kTwoPassMaxThreads && int64_t(nt) * kTwoPassUnroll * 2 < units) nt *= 2;
  const bool causal = q_period > 0;
  const int mode = p.y == nullptr ? kStateOnly : causal ? kProbCausal : p.log_out ? kLogProb : kProb;
  if ((causal && p.log_out) || (p.loss && mode != kStateOnly)) return cudaErrorInvalidValue;
  // [dtype][vec][mode]
  static const RowKernel table[3][2][4] = {
      {{k_twopass<F32, false, kProb>, k_twopass<F32, false, kProbCausal>, k_twopass<F32, false, kLogProb>,
        k_twopass<F32, false, kStateOnly>},
       {k_twopass<F32, true, kProb>, k_twopass<F32, true, kProbCausal>, k_twopass<F32, true, kLogProb>,
        k_twopass<F32, true, kStateOnly>}},
      {{k_twopass<BF16, false, kProb>, k_twopass<BF16, false, kProbCausal>, k_twopass<BF16, false, kLogProb>,
        k_twopass<BF16, false, kStateOnly>},
       {k_twopass<BF16, true, kProb>, k_twopass<BF16, true, kProbCausal>, k_twopass<BF16, true, kLogProb>,
        k_twopass<BF16, true, kStateOnly>}},
      {{k_twopass<F16, false, kProb>, k_twopass<F16, false, kProbCausal>, k_twopass<F16, false, kLogProb>,
        k_twopass<F16, false, kStateOnly>},
       {k_twopass<F16, true, kProb>, k_twopass<F16, true, kProbCausal>, k_twopass<F16, true, kLogProb>,
        k_twopass<F16, true, kStateOnly>}}};
  RowKernel fn = table[p.dtype][vec ? 1 : 0][mode];
  // as the register kernel: up to kGridWaves waves of one-row CTAs before the grid stride
  // (measured: 65536 x 4096 bf16 239 -> 212 us, 262144 x 256 fp32 412 -> 358 us)
  const int64_t cap = int64_t(dev.sm_count) * blocks_per_sm((const void*)fn, nt, 0) * kGridWaves;
  const int grid = int(p.M < cap ? p.M : cap);
  RowArgs a = row_args(p, dev);
  a.q_period = causal ? q_period : 1;
  a.key_offset = key_offset;
  fn<<<grid, nt, 0, p.stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_merge_states(const float* m_a, const float* d_a, const float* m_b,
                                const float* d_b, float* m_out, float* d_out, float* lse_out,
                                int64_t M, cudaStream_t stream, const DeviceInfo& dev) {
  const int64_t want = ceil_div(M, 256);
  const int64_t cap = int64_t(dev.sm_count) * 8;
  const int grid = int(want < cap ? want : cap);
  k_merge_states<<<grid, 256, 0, stream>>>(m_a, d_a, m_b, d_b, m_out, d_out, lse_out, M);
  return cudaGetLastError();
}

}  // namespace rwo
