// kernel_attention.cu -- attention forward with the online softmax: the FlashAttention tile on
// the sm_100 tensor cores (tcgen05).
//
// "从原始Softmax到在线Softmax" derives the blocked form of attention: for query i and key blocks
// j, m' = max(m, max of the block), l = e^(m - m') l + sum e^(s - m'), o~ = e^(m - m') o~ + sum
// e^(s - m') v, o = o~ / l; "5.2 CUDA Online Softmax 实现优化" §8.2 and "Softmax 数值稳定性与
// IO-Aware Attention" §八 describe the same recurrence as FlashAttention, where S = Q K^T never
// leaves the chip.  One CTA owns two tiles of 128 query rows (X = 0, 1) of one head, which take
// turns on the tensor cores: while one tile's softmax runs, the other tile's products run.
//
//  Elements are bf16 or fp16, the head dimension d is 64 or 128.
//  * one producer lane streams Q once and K, V tiles of 128 keys through two shared-memory
//    stages with TMA (cp.async.bulk.tensor, d / 64 boxes of 64 elements x 128 rows per tile with
//    the 128-byte swizzle, zero fill past the sequence end), which lands them directly in the tensor
//    cores' 128-byte-swizzled canonical layouts (Q and K: K-major; V: MN-major, so it needs no
//    transpose); K_j and V_j are issued as soon as their stage is free, each on its own barrier.
//    Rows of 128 bytes per request keep the copy engine and L2 efficient (boxes 16 bytes wide
//    cost one request per 16 bytes and starved the tensor cores);
//  * one thread issues tcgen05.mma (16-bit operands -> fp32, K = 16 per instruction; S: M = N =
//    128; P V: M = 128, N = d) in
//    the order P V_0(j), S_0(j+1), P V_1(j), S_1(j+1): S_X = Q_X K^T into TMEM region S_X, and
//    O_X += P_X V with P_X read from TMEM (A operand in tensor memory); completion is signalled
//    with tcgen05.commit, which covers every earlier product of the thread -- so S_X(j+1) landing
//    also means O_X holds P V_X(j);
//  * two softmax warpgroups, one per query tile: thread t owns query row t (TMEM lane t).  Per key
//    tile it loads its row of S from TMEM, takes the running maximum m (in log2 units of
//    scale * s; moved only when a tile exceeds it by more than 2^8, so O and l are rarely
//    rescaled), rescales its row of O in TMEM by 2^(m_old - m_new) when m moved, and writes
//    P = 2^(s - m) as packed 16-bit values over the first 64 columns of its S region, which the P V
//    product reads.  Masked keys (causal rule, the ragged end of the keys) give P = 0; key tiles
//    wholly above a query tile's causal diagonal are not visited;
//  * epilogue: O / l rounded to the element type, through a per-warp staging buffer and TMA
//    stores, and LSE = m + ln l per row.
// Every wait is bounded (%globaltimer); a wait that runs out sets the status word and the
// kernel still terminates.
//
// Exit drain.  A CTA must not exit while a copy into its shared memory is in flight.  The loader
// lane counts the K and V copies it issues on each stage's barrier; every copy completes one phase
// of its barrier (one arrive with its byte count, then the bytes), in issue order, because a stage
// is refilled only after the product that read its previous tile has finished, and that product
// waited for the tile.  So the last copy on a stage is the stage's n-th phase (n = copies issued
// there) and waiting for the parity of phase n - 1 waits for it, and a phase with the same parity
// two phases back cannot be mistaken for it, since at most one copy per stage is outstanding.  A
// stage with no copy issued is not waited on.  The test hook that skips the first V copy (the
// waits on it run out) is honoured only for at most two key tiles: then each stage receives at
// most one copy, the argument holds as stated, and the skipped copy is simply not counted.
#include <cuda.h>

#include <mutex>

#include "device_common.cuh"
#include "attention.h"
#include "launch.h"

namespace rwo {
namespace {

constexpr int kBM = 128;             // query rows per tile (two tiles per CTA)
constexpr int kBN = 128;             // keys per tile
constexpr int kThreads = 10 * 32;    // 2 x 4 softmax warps, 1 loader warp, 1 MMA warp
constexpr int kLoaderWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;  // S_0 [0, 128), S_1 [128, 256), O_0 [256, 256 + d), O_1 after it
constexpr uint32_t kTmemO = 256;

struct AttnArgs {
  const unsigned char* q;  // [BH][Sq][d] bf16
  const unsigned char* k;  // [BH][Sk][d]
  const unsigned char* v;  // [BH][Sk][d]
  unsigned char* o;        // [BH][Sq][d]
  float* lse;              // [BH][Sq] or null
  int64_t BH, Sq, Sk;
  float c;                 // scale * log2 e
  int causal;
  unsigned* status;
  uint64_t wait_ns;
  int fault;  // test hook (Sk <= 256 only): the first V tile is never copied, so the waits on it run out
};

// Shared memory for head dimension DH (64 or 128), from a 1024-byte aligned base, as the 128-byte
// swizzle needs: Q[2] | K[2] | V[2] | barriers, TMEM address | O staging, 4 KB per softmax warp
// (32 rows x 64 elements, the layout of a 128-byte-swizzled TMA box).
constexpr int kNumBars = 16;
constexpr int kOStage = 32 * 128;
template <int DH>
struct Geo {
  static_assert(DH == 64 || DH == 128, "head dimension 64 or 128");
  static constexpr int kTile = kBN * DH * 2;  // bytes of a Q, K or V tile
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kTile;
  static constexpr int kOffV = 4 * kTile;
  static constexpr int kOffBar = 6 * kTile;
  static constexpr int kOffOStage = kOffBar + 1024;
  static constexpr int kSmem = kOffOStage + 8 * kOStage + 1024;  // + alignment slack
};
static_assert(kNumBars * 8 + 4 <= 1024, "barriers overflow their slot");
// barrier indices
constexpr int kBarQFull = 0, kBarKFull = 1 /*2*/, kBarVFull = 3 /*2*/, kBarKFree = 5 /*2*/, kBarVFree = 7 /*2*/,
              kBarSFull = 9 /*X*/, kBarPFull = 11 /*X*/, kBarODone = 13 /*X*/, kBarQFull1 = 15;

// Q, K and V tiles in shared memory: two blocks of 16 KB (elements 0-63 and 64-127 of each row);
// in a block, row r's 128 bytes at (r / 8) * 1024 + (r % 8) * 128 with its 16-byte chunk c
// stored at chunk position c ^ (r % 8) -- what a TMA box of 64 elements x 128 rows writes with
// the 128-byte swizzle, and the tensor cores' 128-byte-swizzled canonical layout: for Q and K
// (K-major) 8-row groups 1024 B apart (SBO), one MMA's 16 elements of K 32 B further along the
// row; for V (MN-major: rows are keys = K, elements run along N = d) 8-key groups 1024 B apart
// (SBO), the two 64-element halves of N 16 KB apart (LBO), 16 keys per MMA = 2048 B.
//
// P in TMEM (the A operand of P V): row r in lane r, keys 2c and 2c + 1 in column c (low and high
// half), 8 columns per MMA's 16 keys.

// Shared memory matrix descriptor (tcgen05): start >> 4, leading byte offset >> 4, stride byte
// offset >> 4, descriptor version 1, layout (bits 61-63: 0 no swizzle, 2 the 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint64_t layout = 0) {
  return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t(lbo >> 4) << 16) | (uint64_t(sbo >> 4) << 32) | (1ull << 46) |
         (layout << 61);
}
constexpr uint64_t kSw128 = 2;
constexpr uint32_t kBlock = 16384;                                      // one 64-element half of a tile
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

// TMA store of a box (64 elements, 32 rows) from shared memory, and waiting until the copy engine
// has read the staging buffer.
__device__ __forceinline__ void tma_store_box(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y), "r"(z)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_cta() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Instruction descriptor, kind::f16: fp32 accumulator, A and B both bf16 (fmt 1) or both fp16
// (fmt 0), A K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), N columns, M = 128.
__device__ __forceinline__ uint32_t idesc_f16kind(uint32_t fmt, uint32_t b_mn, uint32_t n) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (b_mn << 16) | ((n >> 3) << 17) | ((uint32_t(kBM) >> 4) << 24);
}

// Two fp32 values rounded to the element type (bf16 or fp16), low half first.
template <bool H>
__device__ __forceinline__ uint32_t pack_elem2(float lo, float hi) {
  if constexpr (H) return pack_f16x2(lo, hi);
  else return pack_bf16x2(lo, hi);
}

__device__ __forceinline__ void mma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// A from tensor memory (K-major, two bf16 per column), B from shared memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 64 columns of this warp's 32 TMEM lanes into v (no wait: call tmem_wait_ld before using v).
__device__ __forceinline__ void tmem_ld64_nowait(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Keys i >= vis of a run of 64 keys count as -inf (vis: the row's visible keys from the run's
// start; one 32-bit compare with a constant per key).
__device__ __forceinline__ void mask_keys(uint32_t (&sv)[64], int vis) {
#pragma unroll
  for (int i = 0; i < 64; ++i)
    if (i >= vis) sv[i] = 0xff800000u;
}

// 320 threads, at most 168 registers a thread: three warps share a sub-partition's 16K registers.
// H: fp16 elements (else bf16); DH: head dimension (64 or 128).
template <bool H, int DH>
__global__ void __launch_bounds__(kThreads, 1)
    k_attention_fwd(AttnArgs a, const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tout) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  using GM = Geo<DH>;
  constexpr int kTile = GM::kTile, kOffQ = GM::kOffQ, kOffK = GM::kOffK, kOffV = GM::kOffV, kOffBar = GM::kOffBar,
                kOffOStage = GM::kOffOStage, kD = DH;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffBar + kNumBars * 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto bar = [&](int i) { return smem_addr(&bars[i]); };

  const int64_t ncta = (a.Sq + 2 * kBM - 1) / (2 * kBM);
  // CTA order (launch index L): without a mask, a head's tile pairs side by side while its K and
  // V sit in L2.  Causal: heads in groups of hg (about 128 CTAs a group), and within a group the
  // heaviest pairs (the last rows) of every head first, so the light pairs of one group run beside
  // the heavy pairs of the next and the tail is light, while a group's K and V stay in L2
  // (measured on 128 heads x 16 pairs: groups of 8 heads 0.429 ms; every head's heaviest first
  // across all heads 0.445 ms, with 4x the DRAM traffic; one head after another 0.453 ms).
  int64_t rank, bh;
  {
    const int64_t L = int64_t(blockIdx.y) * gridDim.x + blockIdx.x;
    if (a.causal) {
      const int64_t hg = ncta >= 128 ? 1 : 128 / ncta;
      const int64_t group = L / (hg * ncta), base = group * hg * ncta;
      const int64_t gs = a.BH - group * hg < hg ? a.BH - group * hg : hg;
      rank = (L - base) / gs;
      bh = group * hg + (L - base) % gs;
    } else {
      bh = L / ncta;
      rank = L - bh * ncta;
    }
  }
  const int64_t q0 = (ncta - 1 - rank) * (2 * kBM);
  // key tiles visited by query tile X: all, or (causal, bottom-right aligned) those that hold a
  // key <= the tile's last row + Sk - Sq; none for a tile past the end of the queries
  int nt[2];
  for (int x = 0; x < 2; ++x) {
    const int64_t qx = q0 + x * kBM;
    int64_t kend = qx < a.Sq ? a.Sk : 0;
    if (a.causal && qx < a.Sq) {
      const int64_t last = (qx + kBM - 1 < a.Sq - 1 ? qx + kBM - 1 : a.Sq - 1) + a.Sk - a.Sq + 1;
      kend = last < 0 ? 0 : (last < a.Sk ? last : a.Sk);
    }
    nt[x] = int((kend + kBN - 1) / kBN);
  }
  const int ntmax = nt[0] > nt[1] ? nt[0] : nt[1];

  // The loader lane initialises the barriers and issues the first loads (Q_0 and K_0 first: all
  // that S_0(0) needs) before the block-wide TMEM allocation and barrier.
  const int z = int(bh);
  auto load_tile = [&](const CUtensorMap* map, uint32_t dst, int64_t row0, uint32_t b) {
    for (int c = 0; c < kD / 64; ++c) tma_load_box(dst + uint32_t(c) * kBlock, map, c * 64, int(row0), z, b);
  };
  int nk[2] = {0, 0}, nv[2] = {0, 0};  // K and V copies issued on each stage (loader lane)
  if (warp == kLoaderWarp && lane == 0) {
    mbar_init(bar(kBarQFull), 1);
    mbar_init(bar(kBarQFull1), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(kBarKFull + s), 1);
      mbar_init(bar(kBarVFull + s), 1);
      mbar_init(bar(kBarKFree + s), 1);
      mbar_init(bar(kBarVFree + s), 1);
      mbar_init(bar(kBarSFull + s), 1);
      mbar_init(bar(kBarPFull + s), 4);
      mbar_init(bar(kBarODone + s), 1);
    }
    fence_mbar_init();
    mbar_arrive_expect_tx(bar(kBarQFull), uint32_t(kTile));
    load_tile(&tq, smem_addr(smem + kOffQ), q0, bar(kBarQFull));
    if (ntmax > 0) {
      mbar_arrive_expect_tx(bar(kBarKFull), uint32_t(kTile));
      load_tile(&tk, smem_addr(smem + kOffK), 0, bar(kBarKFull));
      ++nk[0];
    }
    mbar_arrive_expect_tx(bar(kBarQFull1), uint32_t(kTile));
    load_tile(&tq, smem_addr(smem + kOffQ + kTile), q0 + kBM, bar(kBarQFull1));
    if (ntmax > 0 && !a.fault) {
      mbar_arrive_expect_tx(bar(kBarVFull), uint32_t(kTile));
      load_tile(&tv, smem_addr(smem + kOffV), 0, bar(kBarVFull));
      ++nv[0];
    }
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
    // ---- producer: (Q_0, K_0, Q_1, V_0 issued above) K_j, V_j into stage j & 1 ----
    if (lane == 0) {
      for (int j = 1; j < ntmax; ++j) {
        const int s = j & 1;
        const uint32_t par = uint32_t(((j >> 1) - 1) & 1);
        if (j >= 2 && !mbar_wait(bar(kBarKFree + s), par, a.wait_ns)) timed_out = true;  // S(j-2) done
        mbar_arrive_expect_tx(bar(kBarKFull + s), uint32_t(kTile));
        load_tile(&tk, smem_addr(smem + kOffK + s * kTile), int64_t(j) * kBN, bar(kBarKFull + s));
        ++nk[s];
        if (j >= 2 && !mbar_wait(bar(kBarVFree + s), par, a.wait_ns)) timed_out = true;  // P V(j-2) done
        mbar_arrive_expect_tx(bar(kBarVFull + s), uint32_t(kTile));
        load_tile(&tv, smem_addr(smem + kOffV + s * kTile), int64_t(j) * kBN, bar(kBarVFull + s));
        ++nv[s];
      }
      // exit drain: the last copy issued on each stage has landed (see the header)
      for (int s = 0; s < 2; ++s) {
        if (nk[s] > 0 && !mbar_wait(bar(kBarKFull + s), uint32_t((nk[s] - 1) & 1), a.wait_ns)) timed_out = true;
        if (nv[s] > 0 && !mbar_wait(bar(kBarVFull + s), uint32_t((nv[s] - 1) & 1), a.wait_ns)) timed_out = true;
      }
      if (!mbar_wait(bar(kBarQFull), 0u, a.wait_ns)) timed_out = true;
      if (!mbar_wait(bar(kBarQFull1), 0u, a.wait_ns)) timed_out = true;
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer: S_X(0); then per key tile j: P V_0(j), S_0(j+1), P V_1(j), S_1(j+1) ----
    if (lane == 0 && ntmax > 0) {
      const uint32_t fmt = H ? 0u : 1u;
      const uint32_t idS = idesc_f16kind(fmt, 0, uint32_t(kBN)), idPV = idesc_f16kind(fmt, 1, uint32_t(kD));
      auto issue_s = [&](int x, int j) {  // S_x(j) = Q_x K_j^T into S_x; K_j has landed
        const uint32_t sq = smem_addr(smem + kOffQ + x * kTile), sk = smem_addr(smem + kOffK + (j & 1) * kTile);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16(tmem + uint32_t(x * kBN), smem_desc(sq + kmaj_step(kk), 16u, kSwSbo, kSw128),
                   smem_desc(sk + kmaj_step(kk), 16u, kSwSbo, kSw128), idS, kk > 0);
        mma_commit(bar(kBarSFull + x));
      };
      if (!mbar_wait(bar(kBarQFull), 0, a.wait_ns)) timed_out = true;
      if (!mbar_wait(bar(kBarKFull), 0, a.wait_ns)) timed_out = true;
      tc_fence_after();
      if (nt[0] > 0) issue_s(0, 0);
      if (nt[1] > 0) {
        if (!mbar_wait(bar(kBarQFull1), 0, a.wait_ns)) timed_out = true;
        tc_fence_after();
        issue_s(1, 0);
      }
      mma_commit(bar(kBarKFree));
      for (int j = 0; j < ntmax; ++j) {
        const int s = j & 1;
        if (!mbar_wait(bar(kBarVFull + s), uint32_t((j >> 1) & 1), a.wait_ns)) timed_out = true;
        const bool next_k = j + 1 < ntmax;
        bool k_ready = false;
        const uint32_t sv = smem_addr(smem + kOffV + s * kTile);
        for (int x = 0; x < 2; ++x) {
          if (j >= nt[x]) continue;
          if (!mbar_wait(bar(kBarPFull + x), uint32_t(j & 1), a.wait_ns)) timed_out = true;
          tc_fence_after();
          const uint32_t tp = tmem + uint32_t(x * kBN), to = tmem + kTmemO + uint32_t(x * kD);
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            mma_bf16_ts(to, tp + uint32_t(kk) * 8u, smem_desc(sv + kk * kVStep, kBlock, kSwSbo, kSw128), idPV,
                        (j > 0 || kk > 0) ? 1u : 0u);
          if (j + 1 < nt[x]) {
            if (!k_ready) {
              if (!mbar_wait(bar(kBarKFull + (s ^ 1)), uint32_t(((j + 1) >> 1) & 1), a.wait_ns)) timed_out = true;
              tc_fence_after();
              k_ready = true;
            }
            issue_s(x, j + 1);  // overwrites P_x(j) after P V_x(j) has read it (in-order pipe)
          } else {
            mma_commit(bar(kBarODone + x));
          }
        }
        mma_commit(bar(kBarVFree + s));
        if (next_k) mma_commit(bar(kBarKFree + (s ^ 1)));
      }
      // the last commit has arrived before the barriers' memory is released
      const int jl = ntmax - 1;
      if (!mbar_wait(bar(kBarVFree + (jl & 1)), uint32_t((jl >> 1) & 1), a.wait_ns)) timed_out = true;
    }
  } else {
    // ---- softmax warpgroup x: warps 4x .. 4x + 3, thread t = TMEM lane t = query row q0 + 128x + t ----
    const int x = warp >> 2;
    const int t = tid & 127;
    const int ntx = nt[x];
    const int64_t qx = q0 + int64_t(x) * kBM;
    const int64_t qi = qx + t;  // global query row
    const int64_t klim = a.causal ? qi + a.Sk - a.Sq + 1 : a.Sk;  // keys < klim are visible
    // first key at which any row of the tile can be masked (tiles starting past it take the check)
    const int64_t kfull = a.causal ? (qx + a.Sk - a.Sq + 1 < a.Sk ? qx + a.Sk - a.Sq + 1 : a.Sk) : a.Sk;
    const uint32_t lane_base = uint32_t((warp & 3) * 32) << 16;
    const uint32_t ts = tmem + lane_base + uint32_t(x * kBN);
    const uint32_t to = tmem + lane_base + kTmemO + uint32_t(x * kD);
    // running state in log2 units: m = max of c * s (lagging by up to 2^8), l = sum 2^(c s - m)
    constexpr float kSlack = 8.f;
    float m = -INFINITY;
    float l = 0.f;
    for (int j = 0; j < ntx; ++j) {
      if (!mbar_wait(bar(kBarSFull + x), uint32_t(j & 1), a.wait_ns)) timed_out = true;
      tc_fence_after();
      const int64_t k0 = int64_t(j) * kBN;
      // the row maximum, half a row (64 keys) at a time: keys 64-127 first, so that keys 0-63 are
      // still in registers for the exponentials (their P goes over columns 0-31, which they held)
      const bool masked = k0 + kBN > kfull;  // uniform over the warpgroup
      const int vis = int(klim - k0 < 0 ? 0 : klim - k0 > kBN ? kBN : klim - k0);  // visible keys of the tile
      uint32_t sv[64];
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int h = 1 - hh;
        tmem_ld64_nowait(ts + uint32_t(h * 64), sv);
        tmem_wait_ld();
        if (masked) mask_keys(sv, vis - h * 64);
#pragma unroll
        for (int i = 0; i < 64; i += 2) mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], __uint_as_float(sv[i]), __uint_as_float(sv[i + 1]));
      }
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float mtc = __fmul_rn(mt, a.c);
      const bool move = mtc > m + kSlack;  // m = -inf: any visible key moves it
      const float m_new = move ? mtc : m;
      const float alpha = move ? ex2(m - m_new) : 1.f;  // 0 while the row had seen nothing
      const float ms = m_new == -INFINITY ? 0.f : m_new;
      // S_x(j) landing means O_x holds P V_x(j - 1), and P V_x(j) waits for this P: rescale O now
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int h = 0; h < kD / 32; ++h) {  // rare (the maximum moved): 32 columns at a time
          uint32_t ov[32];
          tmem_ld32_nowait(to + h * 32, ov);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__fmul_rn(__uint_as_float(ov[i]), alpha));
          tmem_st32(to + h * 32, ov);
        }
      }
      // P = 2^(c s - m) as packed bf16 over columns 0-63 of S_x (masked keys: 2^-inf = 0); the row
      // sum in fp32, four pairs of partial sums; the exponent by one packed fused multiply-add per pair
      const float2 c2 = make_float2(a.c, a.c), nm2 = make_float2(-ms, -ms);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h == 1) {  // keys 64-127 again (columns 64-127 are untouched by P)
          tmem_ld64_nowait(ts + 64u, sv);
          tmem_wait_ld();
          if (masked) mask_keys(sv, vis - 64);
        }
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float2 t2 = __ffma2_rn(make_float2(__uint_as_float(sv[i]), __uint_as_float(sv[i + 1])), c2, nm2);
          const float2 p = make_float2(ex2(t2.x), ex2(t2.y));
          acc[(i >> 1) & 3] = __fadd2_rn(acc[(i >> 1) & 3], p);
          pk[i >> 1] = pack_elem2<H>(p.x, p.y);
        }
        tmem_st32(ts + uint32_t(h * 32), pk);  // keys 64h .. 64h + 63 -> columns 32h .. 32h + 31
      }
      const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
      const float2 aa = __fadd2_rn(a01, a23);
      l = __fadd_rn(__fmul_rn(l, alpha), __fadd_rn(aa.x, aa.y));
      m = m_new;
      tmem_wait_st();    // P (and O's rescale) in TMEM before the product that reads them
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + x));
    }
    // ---- epilogue: O / l and LSE ----
    if (ntx > 0) {
      if (!mbar_wait(bar(kBarODone + x), 0u, a.wait_ns)) timed_out = true;
      tc_fence_after();
    }
    const float inv = l > 0.f ? __frcp_rn(l) : 0.f;
    // O / l as bf16 through this warp's staging buffer (row = lane, 16-byte chunk c at position
    // c ^ (lane % 8)), one TMA store per 64 columns; rows past Sq are clipped by the copy
    unsigned char* stage = smem + kOffOStage + warp * kOStage;
#pragma unroll 1
    for (int hc = 0; hc < kD / 64; ++hc) {
#pragma unroll 1
      for (int q2 = 0; q2 < 2; ++q2) {
        uint32_t ov[32];
        if (ntx > 0) {
          tmem_ld32_nowait(to + uint32_t(hc * 64 + q2 * 32), ov);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0u;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const float* f = reinterpret_cast<const float*>(ov + 8 * cc);
          uint4 w;
          w.x = pack_elem2<H>(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv));
          w.y = pack_elem2<H>(__fmul_rn(f[2], inv), __fmul_rn(f[3], inv));
          w.z = pack_elem2<H>(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv));
          w.w = pack_elem2<H>(__fmul_rn(f[6], inv), __fmul_rn(f[7], inv));
          const int c = q2 * 4 + cc;
          *reinterpret_cast<uint4*>(stage + lane * 128 + ((c ^ (lane & 7)) << 4)) = w;
        }
      }
      fence_proxy_async_cta();  // the staging writes -> the copy engine
      __syncwarp();
      if (lane == 0) {
        tma_store_box(&tout, smem_addr(stage), hc * 64, int(qx + (warp & 3) * 32), int(bh));
        tma_store_wait_read();  // the buffer is reused (and released at exit) only once read
      }
      __syncwarp();
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

bool attention_fits(int64_t d, int dtype) { return (d == 64 || d == 128) && (dtype == 1 || dtype == 2); }

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

// [BH][S][d] bf16 or fp16, boxes of 64 elements x `rows` rows x 1 head, 128-byte swizzle; rows
// past S read as zeros (loads) or are not written (stores).
bool make_map(CUtensorMap* m, const void* base, int64_t S, int64_t BH, int64_t d, uint32_t rows, bool f16) {
  EncodeTiled fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(S), cuuint64_t(BH)};
  const cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(S) * d * 2};
  const cuuint32_t box[3] = {64, rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attention(const void* q, const void* k, const void* v, void* o, float* lse, int64_t BH, int64_t Sq,
                             int64_t Sk, int64_t d, float scale, bool causal, int dtype, cudaStream_t stream,
                             const DeviceInfo& dev) {
  const bool f16 = dtype == 2;
  using Kern = void (*)(AttnArgs, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap);
  Kern kern = d == 64 ? (f16 ? (Kern)k_attention_fwd<true, 64> : (Kern)k_attention_fwd<false, 64>)
                      : (f16 ? (Kern)k_attention_fwd<true, 128> : (Kern)k_attention_fwd<false, 128>);
  const int smem = d == 64 ? Geo<64>::kSmem : Geo<128>::kSmem;
  cudaError_t err = cudaFuncSetAttribute((const void*)kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  alignas(64) CUtensorMap tq, tk, tv, to;
  if (!make_map(&tq, q, Sq, BH, d, kBM, f16) || !make_map(&tk, k, Sk, BH, d, kBN, f16) ||
      !make_map(&tv, v, Sk, BH, d, kBN, f16) || !make_map(&to, o, Sq, BH, d, 32, f16))
    return cudaErrorInvalidValue;
  AttnArgs a{static_cast<const unsigned char*>(q), static_cast<const unsigned char*>(k),
             static_cast<const unsigned char*>(v), static_cast<unsigned char*>(o), lse, BH, Sq, Sk, scale * kLog2e,
             causal ? 1 : 0, dev.status, exchange_wait_limit_ns(),
             // the skipped-copy test hook only where the exit drain stays exact: two key tiles at most
             debug_fault_attention() && Sk <= 2 * kBN ? 1 : 0};
  const unsigned ncta = unsigned((Sq + 2 * kBM - 1) / (2 * kBM));
  const dim3 grid(ncta, unsigned(BH));
  kern<<<grid, kThreads, smem, stream>>>(a, tq, tk, tv, to);
  return cudaGetLastError();
}

}  // namespace rwo
