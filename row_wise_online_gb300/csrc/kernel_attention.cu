// kernel_attention.cu -- attention forward with the online softmax: the FlashAttention tile on
// the sm_100 tensor cores (tcgen05).
//
// "从原始Softmax到在线Softmax" derives the blocked form of attention: for query i and key blocks
// j, m' = max(m, max of the block), l = e^(m - m') l + sum e^(s - m'), o~ = e^(m - m') o~ + sum
// e^(s - m') v, o = o~ / l; "5.2 CUDA Online Softmax 实现优化" §8.2 and "Softmax 数值稳定性与
// IO-Aware Attention" §八 describe the same recurrence as FlashAttention, where S = Q K^T never
// leaves the chip.  One CTA owns 128 query rows of one head:
//
//  * one producer lane streams Q once and K, V tiles of 128 keys through two shared-memory
//    stages with TMA (cp.async.bulk.tensor, two boxes of 64 elements x 128 rows per tile with the
//    128-byte swizzle, zero fill past the sequence end), which lands them directly in the tensor
//    cores' 128-byte-swizzled canonical layouts (Q and K: K-major; V: MN-major, so it needs no
//    transpose); K_j and V_j are issued as soon as their stage is free, each on its own barrier.
//    Rows of 128 bytes per request keep the copy engine and L2 efficient (boxes 16 bytes wide
//    cost one request per 16 bytes and starved the tensor cores);
//  * one thread issues tcgen05.mma (bf16 x bf16 -> fp32, M = N = 128, K = 16 per instruction):
//    S_j = Q K_j^T into one of two TMEM buffers, so S_{j+1} is computed while S_j is softmaxed,
//    and O += P_j V_j into a third TMEM region; completion is signalled with tcgen05.commit;
//  * four softmax warps: thread t owns query row t (TMEM lane t).  Per tile it loads its row of
//    S from TMEM in one read, takes the running maximum m (in log2 units of scale * s; moved only
//    when a tile exceeds it by more than 2^8, so O and l are rarely rescaled) and, once the
//    previous P V product has landed, rescales the row of O in TMEM by 2^(m_old - m_new), writes
//    P = 2^(s - m) as bf16 into shared memory (the A operand of the P V product) and hands it
//    to the MMA thread.  Masked keys (causal rule, the ragged end of the keys) give P = 0; tiles
//    wholly above the causal diagonal are not visited.
//  * epilogue: O / l as bf16 and LSE = m + ln l per row.
// Every wait is bounded (%globaltimer); a wait that runs out sets the status word and the
// kernel still terminates.
#include <cuda.h>

#include <mutex>

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

// Shared memory (from a 1024-byte aligned base, as the 128-byte swizzle needs):
// Q | K[2] | V[2] | P | barriers | TMEM address.
constexpr int kOffQ = 0;
constexpr int kOffK = kTile;
constexpr int kOffV = 3 * kTile;
constexpr int kOffP = 5 * kTile;
constexpr int kOffBar = 6 * kTile;
constexpr int kNumBars = 14;
constexpr int kSmem = kOffBar + kNumBars * 8 + 16 + 1024;  // + alignment slack
// barrier indices
constexpr int kBarQFull = 0, kBarKFull = 1 /*2*/, kBarVFull = 3 /*2*/, kBarKFree = 5 /*2*/, kBarVFree = 7 /*2*/,
              kBarSFull = 9 /*2*/, kBarPFull = 11, kBarODone = 12;

// Q, K and V tiles in shared memory: two blocks of 16 KB (elements 0-63 and 64-127 of each row);
// in a block, row r's 128 bytes at (r / 8) * 1024 + (r % 8) * 128 with its 16-byte chunk c
// stored at chunk position c ^ (r % 8) -- what a TMA box of 64 elements x 128 rows writes with
// the 128-byte swizzle, and the tensor cores' 128-byte-swizzled canonical layout: for Q and K
// (K-major) 8-row groups 1024 B apart (SBO), one MMA's 16 elements of K 32 B further along the
// row; for V (MN-major: rows are keys = K, elements run along N = d) 8-key groups 1024 B apart
// (SBO), the two 64-element halves of N 16 KB apart (LBO), 16 keys per MMA = 2048 B.
//
// P (written by the softmax threads, no swizzle): 16-byte chunk c (8 keys) of row r at byte
// c * 2048 + r * 16, i.e. K-major core matrices 2048 B apart along K and 128 B apart along M.
__device__ __forceinline__ uint32_t tile_off(int r, int c) { return uint32_t(c * 2048 + r * 16); }

// Shared memory matrix descriptor (tcgen05): start >> 4, leading byte offset >> 4, stride byte
// offset >> 4, descriptor version 1, layout (bits 61-63: 0 no swizzle, 2 the 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint64_t layout = 0) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t(lbo >> 4) << 16) | (uint64_t(sbo >> 4) << 32) | (1ull << 46) |
         (layout << 61);
}
constexpr uint64_t kSw128 = 2;
constexpr uint32_t kBlock = 16384;                                      // one 64-element half of a tile
constexpr uint32_t kPLbo = 2048, kPSbo = 128, kPStep = 4096;            // P, no swizzle: 2 chunks per K step
constexpr uint32_t kSwSbo = 1024;                                       // 8 rows of 128 B
__device__ __forceinline__ uint32_t kmaj_step(int kk) { return uint32_t(kk >> 2) * kBlock + uint32_t(kk & 3) * 32u; }
constexpr uint32_t kVStep = 2048;                                       // 16 keys of V

// TMA: box (64 elements, 128 rows) at (x = element, y = row, z = head) of a [BH][S][128] tensor.
__device__ __forceinline__ void tma_load_box(uint32_t dst, const CUtensorMap* map, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
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

// 64 columns of this warp's 32 TMEM lanes into v (no wait: call tmem_wait_ld before using v).
__device__ __forceinline__ void tmem_ld64_nowait(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
    k_attention_fwd(AttnArgs a, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
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
    mbar_init(bar(kBarQFull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
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
    // ---------------- producer (one lane): TMA loads of Q once, then K_j and V_j ----------------
    if (lane == 0) {
      const int z = int(bh);
      auto load_tile = [&](const CUtensorMap* map, uint32_t dst, int64_t row0, uint32_t b) {
        mbar_arrive_expect_tx(b, uint32_t(kTile));
        for (int c = 0; c < kD / 64; ++c) tma_load_box(dst + uint32_t(c) * kBlock, map, c * 64, int(row0), z, b);
      };
      load_tile(&tq, smem_addr(smem + kOffQ), q0, bar(kBarQFull));
      for (int j = 0; j < nt; ++j) {
        const int s = j & 1;
        const uint32_t par = uint32_t(((j >> 1) - 1) & 1);
        if (j >= 2 && !mbar_wait(bar(kBarKFree + s), par, a.wait_ns)) timed_out = true;  // S_{j-2} done
        load_tile(&tk, smem_addr(smem + kOffK + s * kTile), int64_t(j) * kBN, bar(kBarKFull + s));
        if (j >= 2 && !mbar_wait(bar(kBarVFree + s), par, a.wait_ns)) timed_out = true;  // P V_{j-2} done
        load_tile(&tv, smem_addr(smem + kOffV + s * kTile), int64_t(j) * kBN, bar(kBarVFull + s));
      }
      // every copy has landed before the CTA may exit (the MMA thread normally saw them all)
      for (int j = nt > 2 ? nt - 2 : 0; j < nt; ++j) {
        if (!mbar_wait(bar(kBarKFull + (j & 1)), uint32_t((j >> 1) & 1), a.wait_ns)) timed_out = true;
        if (!mbar_wait(bar(kBarVFull + (j & 1)), uint32_t((j >> 1) & 1), a.wait_ns)) timed_out = true;
      }
      if (nt == 0 && !mbar_wait(bar(kBarQFull), 0u, a.wait_ns)) timed_out = true;
    }
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
          mma_bf16(tmem + uint32_t(s * kBN), smem_desc(sq + kmaj_step(kk), 16u, kSwSbo, kSw128),
                   smem_desc(sk + kmaj_step(kk), 16u, kSwSbo, kSw128), idS, kk > 0);
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
          mma_bf16(tmem + 256u, smem_desc(sp + kk * kPStep, kPLbo, kPSbo),
                   smem_desc(sv + kk * kVStep, kBlock, kSwSbo, kSw128), idPV, (j > 0 || kk > 0) ? 1u : 0u);
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
    // keys below kfull are visible to every row of the tile: tiles under it need no mask
    const int64_t kfull = a.causal ? (q0 + a.Sk - a.Sq + 1 < a.Sk ? q0 + a.Sk - a.Sq + 1 : a.Sk) : a.Sk;
    const uint32_t lane_base = uint32_t(warp * 32) << 16;
    // Running maximum m of c * s (log2 units), moved only when a tile's maximum exceeds it by more
    // than 8: until then P = 2^(c s - m) stays below 2^8 (exact enough in bf16 and fp32) and O, l
    // need no rescale; O / l and LSE = m ln 2 + ln l are the same for any m.
    constexpr float kSlack = 8.f;
    float m = -INFINITY;
    float l = 0.f;
    unsigned char* prow = smem + kOffP;
    for (int j = 0; j < nt; ++j) {
      const int s = j & 1;
      if (!mbar_wait(bar(kBarSFull + s), uint32_t((j >> 1) & 1), a.wait_ns)) timed_out = true;
      tc_fence_after();
      const uint32_t ts = tmem + lane_base + uint32_t(s * kBN);
      const int64_t k0 = int64_t(j) * kBN;
      uint32_t sv[2][64];  // the row of S, one TMEM read
      tmem_ld64_nowait(ts, sv[0]);
      tmem_ld64_nowait(ts + 64, sv[1]);
      tmem_wait_ld();
      const bool masked = k0 + kBN > kfull;  // uniform over the CTA
      if (masked) {  // keys past the row's limit count as -inf
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (k0 + h * 64 + i >= klim) sv[h][i] = 0xff800000u;
      }
      float mx[8];  // eight partial maxima: short dependency chains
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = fmaxf(__uint_as_float(sv[0][i]), __uint_as_float(sv[1][i]));
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 8; i < 64; ++i) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(sv[h][i]));
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float mtc = __fmul_rn(mt, a.c);
      const bool move = mtc > m + kSlack;  // m = -inf: any visible key moves it
      const float m_new = move ? mtc : m;
      const float alpha = move ? ex2(m - m_new) : 1.f;  // 0 while the row had seen nothing
      const float ms = m_new == -INFINITY ? 0.f : m_new;
      // the previous P V product has landed: P's buffer is free and O can be rescaled
      if (j > 0) {
        if (!mbar_wait(bar(kBarODone), uint32_t((j - 1) & 1), a.wait_ns)) timed_out = true;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t to = tmem + lane_base + 256u;
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {  // rare (the maximum moved): half a row at a time
            uint32_t ov[64];
            tmem_ld64_nowait(to + h * 64, ov);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 64; ++i) ov[i] = __float_as_uint(__fmul_rn(__uint_as_float(ov[i]), alpha));
            tmem_st64(to + h * 64, ov);
            tmem_wait_st();
          }
        }
      }
      // P = 2^(c s - m) as bf16 in the A operand layout (masked keys: 2^-inf = 0); the row sum in
      // fp32, four pairs of partial sums; the exponent by one packed fused multiply-add per pair
      const float2 c2 = make_float2(a.c, a.c), nm2 = make_float2(-ms, -ms);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {  // 8 chunks of 8 keys per half
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int i = c8 * 8 + e;
            const float2 t2 = __ffma2_rn(make_float2(__uint_as_float(sv[h][i]), __uint_as_float(sv[h][i + 1])), c2, nm2);
            const float2 p = make_float2(ex2(t2.x), ex2(t2.y));
            acc[e >> 1] = __fadd2_rn(acc[e >> 1], p);
            pk[e >> 1] = pack_bf16x2(p.x, p.y);
          }
          *reinterpret_cast<uint4*>(prow + tile_off(t, h * 8 + c8)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
      const float2 aa = __fadd2_rn(a01, a23);
      l = __fadd_rn(__fmul_rn(l, alpha), __fadd_rn(aa.x, aa.y));
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
    for (int h = 0; h < 2; ++h) {
      uint32_t ov[64];
      if (nt > 0) {
        tmem_ld64_nowait(to + h * 64, ov);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) ov[i] = 0u;
      }
      if (qi < a.Sq) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float* f = reinterpret_cast<const float*>(ov + 8 * q);
          uint4 w;
          w.x = pack_bf16x2(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv));
          w.y = pack_bf16x2(__fmul_rn(f[2], inv), __fmul_rn(f[3], inv));
          w.z = pack_bf16x2(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv));
          w.w = pack_bf16x2(__fmul_rn(f[6], inv), __fmul_rn(f[7], inv));
          *reinterpret_cast<uint4*>(orow + (h * 64 + 8 * q) * 2) = w;
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

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once through the runtime (no link to the driver library).
EncodeTiled encode_tiled() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// [BH][S][128] bf16, boxes of 8 elements x 128 rows x 1 head; rows past S read as zeros.
bool make_map(CUtensorMap* m, const void* base, int64_t S, int64_t BH) {
  EncodeTiled fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cuuint64_t(kD), cuuint64_t(S), cuuint64_t(BH)};
  const cuuint64_t strides[2] = {cuuint64_t(kD) * 2, cuuint64_t(S) * kD * 2};
  const cuuint32_t box[3] = {64, cuuint32_t(kBM), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attention(const void* q, const void* k, const void* v, void* o, float* lse, int64_t BH, int64_t Sq,
                             int64_t Sk, float scale, bool causal, cudaStream_t stream, const DeviceInfo& dev) {
  cudaError_t err = cudaFuncSetAttribute((const void*)k_attention_fwd, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (err != cudaSuccess) return err;
  alignas(64) CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, Sq, BH) || !make_map(&tk, k, Sk, BH) || !make_map(&tv, v, Sk, BH))
    return cudaErrorInvalidValue;
  AttnArgs a{static_cast<const unsigned char*>(q), static_cast<const unsigned char*>(k),
             static_cast<const unsigned char*>(v), static_cast<unsigned char*>(o), lse, Sq, Sk, scale * kLog2e,
             causal ? 1 : 0, dev.status, local_wait_limit_ns()};
  const dim3 grid(unsigned((Sq + kBM - 1) / kBM), unsigned(BH));
  k_attention_fwd<<<grid, kThreads, kSmem, stream>>>(a, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace rwo
