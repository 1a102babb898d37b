// kernel_attention.cu -- attention forward with the online softmax: the FlashAttention tile on
// the sm_100 tensor cores (tcgen05).
//
// "从原始Softmax到在线Softmax" derives the blocked form of attention: for query i and key blocks
// j, m' = max(m, max of the block), l = e^(m - m') l + sum e^(s - m'), o~ = e^(m - m') o~ + sum
// e^(s - m') v, o = o~ / l; "5.2 CUDA Online Softmax 实现优化" §8.2 and "Softmax 数值稳定性与
// IO-Aware Attention" §八 describe the same recurrence as FlashAttention, where S = Q K^T never
// leaves the chip.  One CTA owns 128 query rows of one head:
//
//  * a loader warp streams Q once and K, V tiles of 128 keys through two shared-memory stages
//    with 16-byte cp.async copies placed directly in the tensor cores' no-swizzle canonical
//    layouts (Q and K: K-major core matrices; V: MN-major, so it needs no transpose);
//  * one thread issues tcgen05.mma (bf16 x bf16 -> fp32, M = N = 128, K = 16 per instruction):
//    S_j = Q K_j^T into one of two TMEM buffers, so S_{j+1} is computed while S_j is softmaxed,
//    and O += P_j V_j into a third TMEM region; completion is signalled with tcgen05.commit;
//  * four softmax warps: thread t owns query row t (TMEM lane t).  Per tile it loads its row of
//    S from TMEM, takes the running maximum m (in log2 units of scale * s), rescales l and, once
//    the previous P V product has landed, the row of O in TMEM by 2^(m_old - m_new), writes
//    P = 2^(s - m) as bf16 into shared memory (the A operand of the P V product) and hands it
//    to the MMA thread.  Masked keys (causal rule, the ragged end of the keys) give P = 0; tiles
//    wholly above the causal diagonal are not visited.
//  * epilogue: O / l as bf16 and LSE = m + ln l per row.
// Every wait is bounded (%globaltimer); a wait that runs out sets the status word and the
// kernel still terminates.
#include "device_common.cuh"
#include "launch.h"

namespace rwo {
namespace {

constexpr int kBM = 128;             // query rows per CTA
constexpr int kBN = 128;             // keys per tile
constexpr int kD = 128;              // head dimension
constexpr int kTile = kBN * kD * 2;  // bytes of a K or V tile (and of Q and P)
constexpr int kThreads = 6 * 32;     // 4 softmax warps, 1 loader warp, 1 MMA warp
constexpr int kLoaderWarp = 4;
constexpr int kMmaWarp = 5;
constexpr uint32_t kTmemCols = 512;  // S0 [0, 128), S1 [128, 256), O [256, 384)

struct AttnArgs {
  const unsigned char* q;  // [BH][Sq][d] bf16
  const unsigned char* k;  // [BH][Sk][d]
  const unsigned char* v;  // [BH][Sk][d]
  unsigned char* o;        // [BH][Sq][d]
  float* lse;              // [BH][Sq] or null
  int64_t Sq, Sk;
  float c;                 // scale * log2 e
  int causal;
  unsigned* status;
  uint64_t wait_ns;
};

// Shared memory: Q | K[2] | V[2] | P | barriers | TMEM address.
constexpr int kOffQ = 0;
constexpr int kOffK = kTile;
constexpr int kOffV = 3 * kTile;
constexpr int kOffP = 5 * kTile;
constexpr int kOffBar = 6 * kTile;
constexpr int kNumBars = 14;
constexpr int kSmem = kOffBar + kNumBars * 8 + 16;
// barrier indices
constexpr int kBarQFull = 0, kBarKFull = 1 /*2*/, kBarVFull = 3 /*2*/, kBarKFree = 5 /*2*/, kBarVFree = 7 /*2*/,
              kBarSFull = 9 /*2*/, kBarPFull = 11, kBarODone = 12;

// Byte offset of 16-byte chunk (row r, chunk c) of a K-major tile: core matrices of 8 rows x 16 B,
// consecutive along K (128 B apart), 8-row groups 2048 B apart.
__device__ __forceinline__ uint32_t kmajor_off(int r, int c) { return uint32_t(((r >> 3) * 16 + c) * 128 + (r & 7) * 16); }
// The same for V read as the MN-major B operand: row r = key (K), chunk c = 8 values of d (N).
__device__ __forceinline__ uint32_t mnmajor_off(int r, int c) { return uint32_t((c * 16 + (r >> 3)) * 128 + (r & 7) * 16); }

// Shared memory matrix descriptor (tcgen05): start >> 4, leading byte offset (core-matrix stride
// along K) >> 4, stride byte offset (along M or N) >> 4, descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t(128u >> 4) << 16) | (uint64_t(2048u >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A K-major, B K-major
// (b_mn = 0) or MN-major (b_mn = 1), N = 128, M = 128.
__device__ __forceinline__ uint32_t idesc_bf16(uint32_t b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn << 16) | ((uint32_t(kBN) >> 3) << 17) | ((uint32_t(kBM) >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_cta() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 32 columns of this warp's 32 TMEM lanes: thread `lane` gets lane (32 w + lane), columns col..col+31.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__global__ void __launch_bounds__(kThreads, 1) k_attention_fwd(AttnArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  const int64_t nqt = (a.Sq + kBM - 1) / kBM;
  const int64_t qt = nqt - 1 - int64_t(blockIdx.x);  // the heaviest causal tiles first
  const int64_t bh = blockIdx.y;
  const int64_t q0 = qt * kBM;
  // keys this tile visits: all, or (causal) up to the last row's diagonal
  int64_t kend = a.Sk;
  if (a.causal) {
    const int64_t last = (q0 + kBM - 1 < a.Sq - 1 ? q0 + kBM - 1 : a.Sq - 1) + a.Sk - a.Sq + 1;
    kend = last < 0 ? 0 : (last < a.Sk ? last : a.Sk);
  }
  const int nt = int((kend + kBN - 1) / kBN);

  if (tid == 0) {
    mbar_init(bar(kBarQFull), 32);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarKFull + s), 32);
      mbar_init(bar(kBarVFull + s), 32);
      mbar_init(bar(kBarKFree + s), 1);
      mbar_init(bar(kBarVFree + s), 1);
      mbar_init(bar(kBarSFull + s), 1);
    }
    mbar_init(bar(kBarPFull), 4);
    mbar_init(bar(kBarODone), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool timed_out = false;

  if (warp == kLoaderWarp) {
    // ---------------- loader: Q once, then K and V tiles through two stages ----------------
    const unsigned char* qh = a.q + bh * a.Sq * (kD * 2);
    const unsigned char* kh = a.k + bh * a.Sk * (kD * 2);
    const unsigned char* vh = a.v + bh * a.Sk * (kD * 2);
    const uint32_t sq = smem_addr(smem + kOffQ);
    for (int idx = lane; idx < kBM * 16; idx += 32) {
      const int r = idx >> 4, c = idx & 15;
      if (q0 + r < a.Sq) cp_async16(sq + kmajor_off(r, c), qh + (q0 + r) * (kD * 2) + c * 16);
      else *reinterpret_cast<uint4*>(smem + kOffQ + kmajor_off(r, c)) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
    auto issue_tile = [&](int j) {
      const int s = j & 1;
      const uint32_t sk = smem_addr(smem + kOffK + s * kTile), sv = smem_addr(smem + kOffV + s * kTile);
      for (int idx = lane; idx < kBN * 16; idx += 32) {
        const int r = idx >> 4, c = idx & 15;
        const int64_t key = int64_t(j) * kBN + r;
        if (key < a.Sk) {
          cp_async16(sk + kmajor_off(r, c), kh + key * (kD * 2) + c * 16);
          cp_async16(sv + mnmajor_off(r, c), vh + key * (kD * 2) + c * 16);
        } else {
          *reinterpret_cast<uint4*>(smem + kOffK + s * kTile + kmajor_off(r, c)) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(smem + kOffV + s * kTile + mnmajor_off(r, c)) = make_uint4(0, 0, 0, 0);
        }
      }
      cp_async_commit();
    };
    // The copies of a group are visible to the tensor cores once this thread has waited for the
    // group and fenced the async proxy; then it arrives on the tile's barriers.
    auto land = [&](int j) {
      fence_proxy_async_cta();
      mbar_arrive(bar(kBarKFull + (j & 1)));
      mbar_arrive(bar(kBarVFull + (j & 1)));
    };
    if (nt > 0) issue_tile(0);
    cp_async_wait<1>();  // Q (the groups are Q, then tile 0)
    fence_proxy_async_cta();
    mbar_arrive(bar(kBarQFull));
    int landed = -1;  // last tile handed over
    for (int j = 1; j < nt; ++j) {
      if (j == 1) {
        issue_tile(1);
        cp_async_wait<1>();  // tile 0 has landed (tile 1 may still be in flight)
        land(0);
        landed = 0;
      } else {
        // Hand tile j - 1 over before waiting for stage j & 1: the products that free the stage
        // (S_{j-2}, P_{j-2} V_{j-2}) come after S_{j-1} in the MMA thread's order.
        cp_async_wait<0>();
        land(j - 1);
        landed = j - 1;
        const uint32_t par = uint32_t(((j >> 1) - 1) & 1);
        if (!mbar_wait(bar(kBarKFree + (j & 1)), par, a.wait_ns)) timed_out = true;
        if (!mbar_wait(bar(kBarVFree + (j & 1)), par, a.wait_ns)) timed_out = true;
        issue_tile(j);
      }
    }
    cp_async_wait<0>();
    for (int j = landed + 1; j < nt; ++j) land(j);
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issue (one thread) ----------------
    if (lane == 0) {
      const uint32_t idS = idesc_bf16(0), idPV = idesc_bf16(1);
      const uint32_t sq = smem_addr(smem + kOffQ), sp = smem_addr(smem + kOffP);
      auto issue_s = [&](int j) {
        const int s = j & 1;
        if (!mbar_wait(bar(kBarKFull + s), uint32_t((j >> 1) & 1), a.wait_ns)) timed_out = true;
        tc_fence_after();
        const uint32_t sk = smem_addr(smem + kOffK + s * kTile);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16(tmem + uint32_t(s * kBN), smem_desc(sq + kk * 256), smem_desc(sk + kk * 256), idS, kk > 0);
        mma_commit(bar(kBarSFull + s));
        mma_commit(bar(kBarKFree + s));
      };
      if (!mbar_wait(bar(kBarQFull), 0, a.wait_ns)) timed_out = true;
      if (nt > 0) issue_s(0);
      if (nt > 1) issue_s(1);
      for (int j = 0; j < nt; ++j) {
        // P_j written (and S_j read, and O rescaled) by the softmax warps
        if (!mbar_wait(bar(kBarPFull), uint32_t(j & 1), a.wait_ns)) timed_out = true;
        if (!mbar_wait(bar(kBarVFull + (j & 1)), uint32_t((j >> 1) & 1), a.wait_ns)) timed_out = true;
        tc_fence_after();
        const uint32_t sv = smem_addr(smem + kOffV + (j & 1) * kTile);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_bf16(tmem + 256u, smem_desc(sp + kk * 256), smem_desc(sv + kk * 256), idPV, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(bar(kBarODone));
        mma_commit(bar(kBarVFree + (j & 1)));
        if (j + 2 < nt) issue_s(j + 2);  // S buffer j & 1 was read before P_j was handed over
      }
    }
  } else {
    // ---------------- softmax warps: thread t owns query row t ----------------
    const int t = tid;                 // 0..127, TMEM lane t
    const int64_t qi = q0 + t;         // global query row
    const int64_t klim = a.causal ? qi + a.Sk - a.Sq + 1 : a.Sk;  // keys < klim are visible
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    float m = -INFINITY;  // running maximum of c * s (log2 units)
    float l = 0.f;
    unsigned char* prow = smem + kOffP;
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1;
      if (!mbar_wait(bar(kBarSFull + s), uint32_t((j >> 1) & 1), a.wait_ns)) timed_out = true;
      tc_fence_after();
      const uint32_t ts = tmem + lane_base + uint32_t(s * kBN);
      const int64_t k0 = int64_t(j) * kBN;
      // the row's maximum over this tile (masked keys excluded)
      float mt = -INFINITY;
#pragma unroll 1
      for (int c0 = 0; c0 < kBN; c0 += 32) {
        float sv[32];
        tmem_ld32(ts + c0, sv);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (k0 + c0 + i < klim) mt = fmaxf(mt, sv[i]);
      }
      const float m_new = fmaxf(m, __fmul_rn(mt, a.c));
      const float ms = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2(m - ms);  // 0 while the row has seen nothing
      // the previous P V product has landed: P's buffer is free and O can be rescaled
      if (j > 0) {
        if (!mbar_wait(bar(kBarODone), uint32_t((j - 1) & 1), a.wait_ns)) timed_out = true;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t to = tmem + lane_base + 256u;
#pragma unroll 1
          for (int c0 = 0; c0 < kD; c0 += 32) {
            float ov[32];
            tmem_ld32(to + c0, ov);
#pragma unroll
            for (int i = 0; i < 32; ++i) ov[i] = __fmul_rn(ov[i], alpha);
            tmem_st32(to + c0, ov);
          }
        }
      }
      // P = 2^(c s - m) as bf16 in the A operand layout; the row sum in fp32
      float sum = 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < kBN; c0 += 32) {
        float sv[32];
        tmem_ld32(ts + c0, sv);
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float p0 = k0 + c0 + i < klim ? ex2(__fsub_rn(__fmul_rn(sv[i], a.c), ms)) : 0.f;
          const float p1 = k0 + c0 + i + 1 < klim ? ex2(__fsub_rn(__fmul_rn(sv[i + 1], a.c), ms)) : 0.f;
          sum += p0 + p1;
          pk[i >> 1] = pack_bf16x2(p0, p1);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4*>(prow + kmajor_off(t, (c0 >> 3) + q)) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      l = __fadd_rn(__fmul_rn(l, alpha), sum);
      m = m_new;
      fence_proxy_async_cta();  // P's generic stores -> the tensor cores' async proxy
      tc_fence_before();        // O's TMEM stores before the next product
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull));
    }
    // epilogue: O / l, LSE = m ln 2 + ln l
    if (nt > 0) {
      if (!mbar_wait(bar(kBarODone), uint32_t((nt - 1) & 1), a.wait_ns)) timed_out = true;
      tc_fence_after();
    }
    const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
    const uint32_t to = tmem + lane_base + 256u;
    unsigned char* orow = a.o + (bh * a.Sq + qi) * (kD * 2);
#pragma unroll 1
    for (int c0 = 0; c0 < kD; c0 += 32) {
      float ov[32];
      if (nt > 0) {
        tmem_ld32(to + c0, ov);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) ov[i] = 0.f;
      }
      if (qi < a.Sq) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w;
          w.x = pack_bf16x2(__fmul_rn(ov[8 * q + 0], inv), __fmul_rn(ov[8 * q + 1], inv));
          w.y = pack_bf16x2(__fmul_rn(ov[8 * q + 2], inv), __fmul_rn(ov[8 * q + 3], inv));
          w.z = pack_bf16x2(__fmul_rn(ov[8 * q + 4], inv), __fmul_rn(ov[8 * q + 5], inv));
          w.w = pack_bf16x2(__fmul_rn(ov[8 * q + 6], inv), __fmul_rn(ov[8 * q + 7], inv));
          *reinterpret_cast<uint4*>(orow + (c0 + 8 * q) * 2) = w;
        }
      }
    }
    if (qi < a.Sq && a.lse)
      a.lse[bh * a.Sq + qi] = l > 0.f ? __fadd_rn(__fmul_rn(m, 0.6931471805599453f), logf(l)) : -INFINITY;
  }
  if (timed_out && lane == 0) atomicOr(a.status, kStatusTimeout);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
}

}  // namespace

bool attention_fits(int64_t d, int dtype) { return d == kD && dtype == 1; }

cudaError_t launch_attention(const void* q, const void* k, const void* v, void* o, float* lse, int64_t BH, int64_t Sq,
                             int64_t Sk, float scale, bool causal, cudaStream_t stream, const DeviceInfo& dev) {
  cudaError_t err = cudaFuncSetAttribute((const void*)k_attention_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err != cudaSuccess) return err;
  AttnArgs a{static_cast<const unsigned char*>(q), static_cast<const unsigned char*>(k),
             static_cast<const unsigned char*>(v), static_cast<unsigned char*>(o), lse, Sq, Sk, scale * kLog2e,
             causal ? 1 : 0, dev.status, local_wait_limit_ns()};
  const dim3 grid(unsigned((Sq + kBM - 1) / kBM), unsigned(BH));
  k_attention_fwd<<<grid, kThreads, kSmem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace rwo
