// device_common.cuh -- device primitives shared by the row-wise online softmax kernels.
//
// * State / merge: the online (m, d) state and its merge ("5.2 CUDA Online Softmax
//   实现优化", §2.1 and §4.1; "Softmax 数值稳定性与 IO-Aware Attention", §4.1), with the
//   empty state (-inf, 0) as identity: the exponent offset uses m_safe = 0 when m = -inf,
//   so ex2(-inf - 0) = 0 replaces the NaN of -inf - (-inf).
// * Exponentials are ex2.approx.ftz.f32 of (a - b) * log2(e): the difference is formed
//   first so the rounding error scales with the spread of the row, not its magnitude.
// * Warp (butterfly) and block (shared memory) merges ("5.2 ..." §4.2; "Softmax 数值稳定性
//   ..." §4.2).  The merge is written to be bit-symmetric, so every lane of a butterfly and
//   every warp of a block ends with the identical state.
// * bf16 <-> fp32 conversion, 16-byte vector I/O.
// * Inline-PTX wrappers for mbarrier, cp.async.bulk (global <-> shared), proxy fences,
//   L2 cache policies, DSMEM and %globaltimer, used by the bulk-copy kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace rwo {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------------------------
// Arithmetic
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// e^(c (a - b) / log2 e) for b finite (b is an m_safe); a = -inf gives 0.  c = log2 e gives
// e^(a - b); c = scale * log2 e gives e^(scale (a - b)), the softmax of scale * x.
__device__ __forceinline__ float exp_diff(float a, float b, float c = kLog2e) {
  return ex2(__fmul_rn(__fsub_rn(a, b), c));
}

// The same for a pair of values, with the shift passed negated.  The packed f32x2 add and
// multiply of sm_100 and later round each half exactly as the scalar instructions do, so this
// gives bit for bit the two exp_diff values in half the add/multiply issue slots.
__device__ __forceinline__ float2 exp_diff2(float2 a, float2 neg_b, float c = kLog2e) {
  const float2 t = __fmul2_rn(__fadd2_rn(a, neg_b), make_float2(c, c));
  return make_float2(ex2(t.x), ex2(t.y));
}

__device__ __forceinline__ float safe_max(float m) { return m == -INFINITY ? 0.f : m; }

// Sum of e^(x - m) over pairs, with one packed fused multiply-add per pair for the exponent:
// fma(x, log2 e, -mc) where mc = m log2 e rounded.  The exact value of that fma is
// (x - m) log2 e + delta with delta = m log2 e - mc, the same for every term, so the sum comes
// out scaled by 2^delta; delta is exact (fma(m, log2 e, -mc)) and the scale is removed at the
// end.  Only for |m| < 2^20, where |delta| <= 1/16 and 2^-delta is accurate; the caller uses
// the difference form (exp_diff2) otherwise.  m must be an m_safe (finite).
struct ExpShift {
  float2 log2e2, neg_mc2;
  float unscale;  // 2^-delta
};
__device__ __forceinline__ ExpShift exp_shift(float m, float c = kLog2e) {
  const float mc = __fmul_rn(m, c);
  const float delta = __fmaf_rn(m, c, -mc);
  return ExpShift{make_float2(c, c), make_float2(-mc, -mc), ex2(-delta)};
}
__device__ __forceinline__ float2 exp_shifted2(float2 x, const ExpShift& s) {
  const float2 t = __ffma2_rn(x, s.log2e2, s.neg_mc2);
  return make_float2(ex2(t.x), ex2(t.y));
}
__device__ __forceinline__ bool exp_shift_ok(float m) { return fabsf(m) < 0x1p20f; }

struct State {
  float m;  // running maximum (raw input units)
  float d;  // sum of e^(x - m) over the folded elements
};

__device__ __forceinline__ State empty_state() { return State{-INFINITY, 0.f}; }

// Merge of two partial states.  Each product is rounded on its own before the add, so
// merge(a, b) and merge(b, a) are bitwise equal.
__device__ __forceinline__ State merge(State a, State b, float c = kLog2e) {
  const float m = fmaxf(a.m, b.m);
  const float ms = safe_max(m);
  const float sa = exp_diff(a.m, ms, c);
  const float sb = exp_diff(b.m, ms, c);
  return State{m, __fadd_rn(__fmul_rn(a.d, sa), __fmul_rn(b.d, sb))};
}

// Butterfly merge over the 32 lanes of a warp; every lane returns the same state.
__device__ __forceinline__ State warp_merge(State s, float c = kLog2e) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    State t;
    t.m = __shfl_xor_sync(0xffffffffu, s.m, o);
    t.d = __shfl_xor_sync(0xffffffffu, s.d, o);
    s = merge(s, t, c);
  }
  return s;
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Merge across the `nwarps` warps taking part (warp index `warp`, lane `lane`).  `slots`
// points at nwarps State entries of shared memory reserved for this call (callers alternate
// two buffers between consecutive rows, so one barrier per row suffices).  `sync()` is the
// barrier over exactly those warps.  Every participating thread returns the same state.
template <class Sync>
__device__ __forceinline__ State group_merge(State s, State* slots, int nwarps, int warp, int lane,
                                             Sync sync, float c = kLog2e) {
  s = warp_merge(s, c);
  if (nwarps == 1) return s;
  if (lane == 0) slots[warp] = s;
  sync();
  // Lanes hold the warp states replicated modulo p (the power of two >= nwarps), so a butterfly
  // over offsets p/2 .. 1 leaves the full merge in every lane: log2(p) rounds instead of 5.
  int p = 1;
  while (p < nwarps) p <<= 1;
  const int i = lane & (p - 1);
  State t = i < nwarps ? slots[i] : empty_state();
  for (int o = p >> 1; o > 0; o >>= 1) {
    State u;
    u.m = __shfl_xor_sync(0xffffffffu, t.m, o);
    u.d = __shfl_xor_sync(0xffffffffu, t.d, o);
    t = merge(t, u, c);
  }
  return t;
}

// The same merges taken n-ary instead of pairwise: m = max_i m_i first (a max butterfly), then
// d = sum_i d_i e^(m_i - m) (one rescale per lane, a sum butterfly).  This is the merge formula
// applied to all parts at once -- equal to the pairwise tree up to the order of the additions --
// at one exponential per lane instead of two per round.
__device__ __forceinline__ State warp_merge_nary(State s, float c = kLog2e) {
  float m = s.m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float d = __fmul_rn(s.d, exp_diff(s.m, safe_max(m), c));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) d = __fadd_rn(d, __shfl_xor_sync(0xffffffffu, d, o));
  return State{m, d};
}

template <class Sync>
__device__ __forceinline__ State group_merge_nary(State s, State* slots, int nwarps, int warp, int lane,
                                                  Sync sync, float c = kLog2e) {
  s = warp_merge_nary(s, c);
  if (nwarps == 1) return s;
  if (lane == 0) slots[warp] = s;
  sync();
  int p = 1;
  while (p < nwarps) p <<= 1;
  const int i = lane & (p - 1);
  const State t = i < nwarps ? slots[i] : empty_state();
  float m = t.m;
  for (int o = p >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float d = __fmul_rn(t.d, exp_diff(t.m, safe_max(m), c));
  for (int o = p >> 1; o > 0; o >>= 1) d = __fadd_rn(d, __shfl_xor_sync(0xffffffffu, d, o));
  return State{m, d};
}

// 1/d, with 0 for an empty row (d = 0) so that y = 0 there instead of 0 * inf.
__device__ __forceinline__ float safe_inv(float d) { return d > 0.f ? __frcp_rn(d) : 0.f; }

__device__ __forceinline__ float lse_of(State s) {
  return s.m == -INFINITY ? -INFINITY : s.m + logf(s.d);
}

// log y_j = x_j - LSE, evaluated as (x_j - m) - ln d: the difference x_j - m is exact for the
// entries near the maximum (the ones that matter), so only ln d and the last subtraction round.
// An empty row (d = 0) gives ln d = +inf, so every entry becomes -inf (log 0).
struct LogNorm {
  float ms;   // m_safe
  float lnd;  // ln d
};
__device__ __forceinline__ LogNorm log_norm(State s) {
  return LogNorm{safe_max(s.m), s.d > 0.f ? logf(s.d) : INFINITY};
}
// With a scale (the softmax of scale * x, m the raw maximum): scale (x - m) - ln d, one rounding
// for the product and the subtraction (identical to the unscaled form when scale = 1).
__device__ __forceinline__ float log_prob(float x, LogNorm n, float scale = 1.f) {
  return __fmaf_rn(__fsub_rn(x, n.ms), scale, -n.lnd);
}

// The state reported for the softmax of scale * x: m scaled (monotone rounding keeps it the
// maximum of the rounded scale * x_j), d unchanged (already relative to it).
__device__ __forceinline__ State scaled_state(State s, float scale) { return State{__fmul_rn(s.m, scale), s.d}; }

// Cross-entropy loss -log p_label = (m - x_label) + ln d, in the order the page's
// cross_entropy_loss takes it (logits - max first): m - x_label is exact when the two are close,
// so a large |m| costs no cancellation, as LSE - x_label would.  An all -inf row gives NaN.
__device__ __forceinline__ float ce_loss(State s, float x_label, float scale = 1.f) {
  if (s.m == -INFINITY) return __int_as_float(0x7fc00000);
  return __fmaf_rn(__fsub_rn(s.m, x_label), scale, logf(s.d));
}

// ---------------------------------------------------------------------------------------------
// Element types
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two fp32 -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint16_t to_bf16(float v) {
  uint16_t r;
  asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(r) : "f"(v));
  return r;
}

struct F32 {
  static constexpr int kVec = 4;    // elements per 16-byte vector
  static constexpr int kBytes = 4;  // bytes per element
  static constexpr uint32_t kNegInfWord = 0xff800000u;
  __device__ static __forceinline__ void unpack(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ uint4 pack(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                      __float_as_uint(f[3]));
  }
  __device__ static __forceinline__ void unpack2(const uint4& v, float2 (&f)[2]) {
    f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  __device__ static __forceinline__ uint4 pack2(const float2 (&f)[2]) {
    return make_uint4(__float_as_uint(f[0].x), __float_as_uint(f[0].y), __float_as_uint(f[1].x),
                      __float_as_uint(f[1].y));
  }
  __device__ static __forceinline__ float load1(const void* p, int64_t i) {
    return __ldg(static_cast<const float*>(p) + i);
  }
  // Element i of a row staged in shared memory at address `slot`.
  __device__ static __forceinline__ float lds1(uint32_t slot, int64_t i) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(slot + uint32_t(i) * 4u) : "memory");
    return v;
  }
  // Largest of the vector's four values.
  __device__ static __forceinline__ float vmax(const uint4& v) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                 fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  }
  // Largest value of n vectors.
  template <int n>
  __device__ static __forceinline__ float vmax_all(const uint4 (&q)[n]) {
    float m = vmax(q[0]);
#pragma unroll
    for (int k = 1; k < n; ++k) m = fmaxf(m, vmax(q[k]));
    return m;
  }
  __device__ static __forceinline__ void store1(void* p, int64_t i, float v) {
    static_cast<float*>(p)[i] = v;
  }
};

struct BF16 {
  static constexpr int kVec = 8;
  static constexpr int kBytes = 2;
  static constexpr uint32_t kNegInfWord = 0xff80ff80u;
  __device__ static __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
    f[0] = bf16_lo(v.x);
    f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y);
    f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z);
    f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w);
    f[7] = bf16_hi(v.w);
  }
  __device__ static __forceinline__ uint4 pack(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
  }
  __device__ static __forceinline__ void unpack2(const uint4& v, float2 (&f)[4]) {
    f[0] = make_float2(bf16_lo(v.x), bf16_hi(v.x));
    f[1] = make_float2(bf16_lo(v.y), bf16_hi(v.y));
    f[2] = make_float2(bf16_lo(v.z), bf16_hi(v.z));
    f[3] = make_float2(bf16_lo(v.w), bf16_hi(v.w));
  }
  __device__ static __forceinline__ uint4 pack2(const float2 (&f)[4]) {
    return make_uint4(pack_bf16x2(f[0].x, f[0].y), pack_bf16x2(f[1].x, f[1].y), pack_bf16x2(f[2].x, f[2].y),
                      pack_bf16x2(f[3].x, f[3].y));
  }
  __device__ static __forceinline__ float load1(const void* p, int64_t i) {
    const unsigned short b = __ldg(static_cast<const unsigned short*>(p) + i);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  __device__ static __forceinline__ float lds1(uint32_t slot, int64_t i) {
    unsigned short b;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(b) : "r"(slot + uint32_t(i) * 2u) : "memory");
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  // Largest of the vector's eight values: packed bf16x2 max (exact), then one widening.
  __device__ static __forceinline__ float vmax(const uint4& v) {
    uint32_t a, b, m;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z), "r"(v.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
    return fmaxf(bf16_lo(m), bf16_hi(m));
  }
  // Largest value of n vectors: a packed bf16x2 max over all their words, then one widening.
  template <int n>
  __device__ static __forceinline__ float vmax_all(const uint4 (&q)[n]) {
    uint32_t w[4] = {q[0].x, q[0].y, q[0].z, q[0].w};
#pragma unroll
    for (int k = 1; k < n; ++k) {
      asm("max.bf16x2 %0, %0, %1;" : "+r"(w[0]) : "r"(q[k].x));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(w[1]) : "r"(q[k].y));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(w[2]) : "r"(q[k].z));
      asm("max.bf16x2 %0, %0, %1;" : "+r"(w[3]) : "r"(q[k].w));
    }
    return vmax(make_uint4(w[0], w[1], w[2], w[3]));
  }
  __device__ static __forceinline__ void store1(void* p, int64_t i, float v) {
    static_cast<uint16_t*>(p)[i] = to_bf16(v);
  }
};

// IEEE binary16: conversions by cvt (exact widening, round-to-nearest-even narrowing, subnormals
// kept), packed max.f16x2 for the maximum.
__device__ __forceinline__ float f16_lo(uint32_t w) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(w));
  return f;
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(w));
  return f;
}
// Two fp32 -> packed f16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

struct F16 {
  static constexpr int kVec = 8;
  static constexpr int kBytes = 2;
  static constexpr uint32_t kNegInfWord = 0xfc00fc00u;
  __device__ static __forceinline__ void unpack(const uint4& v, float (&f)[8]) {
    f[0] = f16_lo(v.x);
    f[1] = f16_hi(v.x);
    f[2] = f16_lo(v.y);
    f[3] = f16_hi(v.y);
    f[4] = f16_lo(v.z);
    f[5] = f16_hi(v.z);
    f[6] = f16_lo(v.w);
    f[7] = f16_hi(v.w);
  }
  __device__ static __forceinline__ uint4 pack(const float (&f)[8]) {
    return make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                      pack_f16x2(f[6], f[7]));
  }
  __device__ static __forceinline__ void unpack2(const uint4& v, float2 (&f)[4]) {
    f[0] = make_float2(f16_lo(v.x), f16_hi(v.x));
    f[1] = make_float2(f16_lo(v.y), f16_hi(v.y));
    f[2] = make_float2(f16_lo(v.z), f16_hi(v.z));
    f[3] = make_float2(f16_lo(v.w), f16_hi(v.w));
  }
  __device__ static __forceinline__ uint4 pack2(const float2 (&f)[4]) {
    return make_uint4(pack_f16x2(f[0].x, f[0].y), pack_f16x2(f[1].x, f[1].y), pack_f16x2(f[2].x, f[2].y),
                      pack_f16x2(f[3].x, f[3].y));
  }
  __device__ static __forceinline__ float load1(const void* p, int64_t i) {
    const unsigned short b = __ldg(static_cast<const unsigned short*>(p) + i);
    return f16_lo(b);
  }
  __device__ static __forceinline__ float lds1(uint32_t slot, int64_t i) {
    unsigned short b;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(b) : "r"(slot + uint32_t(i) * 2u) : "memory");
    return f16_lo(b);
  }
  // Largest of the vector's eight values: packed f16x2 max (exact), then one widening.
  __device__ static __forceinline__ float vmax(const uint4& v) {
    uint32_t a, b, m;
    asm("max.f16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
    asm("max.f16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z), "r"(v.w));
    asm("max.f16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
    return fmaxf(f16_lo(m), f16_hi(m));
  }
  template <int n>
  __device__ static __forceinline__ float vmax_all(const uint4 (&q)[n]) {
    uint32_t w[4] = {q[0].x, q[0].y, q[0].z, q[0].w};
#pragma unroll
    for (int k = 1; k < n; ++k) {
      asm("max.f16x2 %0, %0, %1;" : "+r"(w[0]) : "r"(q[k].x));
      asm("max.f16x2 %0, %0, %1;" : "+r"(w[1]) : "r"(q[k].y));
      asm("max.f16x2 %0, %0, %1;" : "+r"(w[2]) : "r"(q[k].z));
      asm("max.f16x2 %0, %0, %1;" : "+r"(w[3]) : "r"(q[k].w));
    }
    return vmax(make_uint4(w[0], w[1], w[2], w[3]));
  }
  __device__ static __forceinline__ void store1(void* p, int64_t i, float v) {
    static_cast<uint16_t*>(p)[i] = uint16_t(pack_f16x2(v, 0.f) & 0xffffu);
  }
};

// Keep the first `keep` (0 < keep < kVec) elements of a packed vector and set the rest to -inf.
template <class D>
__device__ __forceinline__ uint4 mask_tail(uint4 v, int keep) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
  constexpr int per_word = 4 / D::kBytes;  // elements per 32-bit word
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (per_word == 1) {
      if (i >= keep) w[i] = 0xff800000u;
    } else {
      if (2 * i >= keep) w[i] = D::kNegInfWord;
      else if (2 * i + 1 >= keep) w[i] = (w[i] & 0x0000ffffu) | (D::kNegInfWord & 0xffff0000u);  // high half: 2i+1
    }
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------------------------------------
// 16-byte global memory access
// ---------------------------------------------------------------------------------------------

// Read-only streaming load (input read once): no L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Plain coherent 16-byte load (used where the same lines are read twice).
__device__ __forceinline__ uint4 ld16(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Streaming store (output written once, not re-read by this kernel).
__device__ __forceinline__ void st_stream16(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------------------------
// Shared memory, mbarrier and bulk copies (sm_90+ PTX; used on sm_103a)
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds16(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy and to the cluster.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `parity` of a local mbarrier to complete, for at most
// `limit_ns` nanoseconds.  Returns false if the limit ran out (the caller records it).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Bulk copy global -> shared (this CTA), completion signalled on mbarrier `bar` as
// transaction bytes.  src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                        uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Bulk copy shared (this CTA) -> global, tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes, uint64_t policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
               "r"(src), "r"(bytes), "l"(policy)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// All committed bulk stores of this thread have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// All committed bulk stores of this thread are complete (written to global memory).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------------------------------------
// Thread-block clusters and distributed shared memory
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// The shared::cluster address of `local` in the CTA of rank `rank` of this cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

// Arrive on an mbarrier in another CTA of the cluster, releasing this thread's prior
// (distributed) shared memory writes to the waiter.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// ---------------------------------------------------------------------------------------------
// Global-memory release/acquire (cross-cluster exchange)
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

}  // namespace rwo
