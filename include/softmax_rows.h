/*
 * softmax_rows.h -- C ABI of the GB300 (sm_103a) row-wise online softmax library.
 *
 * Library: row_wise_online_gb300/lib/libsoftmax_rows.so.  Every compute call
 * enqueues CUDA kernels on the caller's stream and returns at once; every step
 * of the computation runs in the library's own kernels.
 *
 * The problem (as stated on "5.2 CUDA Online Softmax 实现优化", §1.1 and
 * §2): for each row r of a row-major M x N matrix x,
 *
 *     m_r   = max_j x[r, j]
 *     d_r   = sum_j exp(x[r, j] - m_r)
 *     y[r,j]= exp(x[r, j] - m_r) / d_r
 *     LSE_r = m_r + ln d_r      ("从原始Softmax到在线Softmax", log-sum-exp)
 *
 * computed with the online (m, d) recurrence (§2.1 of the same page): each
 * thread folds its elements into a running max and a rescaled exp-sum, and
 * partial states are merged with m = max(m1, m2),
 * d = d1 e^(m1 - m) + d2 e^(m2 - m)  (§4.1; "Softmax 数值稳定性与 IO-Aware
 * Attention" §4.1).  The empty state (-inf, 0) is the identity of that merge,
 * so a fully masked (-inf) chunk, thread, warp or block contributes nothing
 * and never produces NaN.  A row whose entries are all -inf gives y = 0,
 * m = -inf, d = 0, LSE = -inf.
 *
 * Conventions shared by every call:
 *  - Pointers are DEVICE pointers (except softmax_rows_host), owned by the
 *    caller; the library keeps none of them after the call is enqueued.
 *  - Matrices are row-major and contiguous: row r starts at element r * N.
 *  - dtype is SOFTMAX_F32 (fp32 in / fp32 out), SOFTMAX_BF16 (bf16 bit
 *    patterns in / bf16 out) or SOFTMAX_F16 (IEEE binary16 in / out); 16-bit
 *    outputs are rounded to nearest even (fp16 keeps subnormals).  Arithmetic
 *    is fp32 in every case; exponentials use the hardware ex2 with a log2(e)
 *    prescale.  fp16's range ends at 65504 ("Softmax 数值稳定性与 IO-Aware
 *    Attention" §一, precision and range of the floating-point formats):
 *    inputs cannot exceed it, softmax outputs (in [0, 1]) always fit, and
 *    log-softmax outputs below -65504 round to -inf.
 *  - State outputs m_out, d_out, lse_out are fp32 arrays of M entries; each
 *    may be NULL.  m_out is the raw row maximum (bit-exact max of the inputs,
 *    -0 and +0 equal).  d_out is relative to m_out, natural base.
 *  - stream is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *  - M == 0 is a no-op returning SOFTMAX_OK (the pointers may then be NULL,
 *    as they are for an empty tensor); N, dtype and variant are still checked.
 *  - Return value: a softmax_status.  Argument errors are detected on the
 *    host before anything is enqueued.  A CUDA launch error returns
 *    SOFTMAX_ERR_CUDA (softmax_last_cuda_error() names it).  Errors found by a
 *    kernel while it runs (a bounded wait that ran out) are recorded in a
 *    per-device status word read by softmax_get_status().
 */
#ifndef ROW_WISE_ONLINE_SOFTMAX_ROWS_H
#define ROW_WISE_ONLINE_SOFTMAX_ROWS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
enum softmax_dtype { SOFTMAX_F32 = 0, SOFTMAX_BF16 = 1, SOFTMAX_F16 = 2 };

/* Status codes. */
enum softmax_status {
  SOFTMAX_OK = 0,
  SOFTMAX_ERR_INVALID_ARG = 1, /* NULL pointer, N < 1, M < 0, unknown dtype/variant, size overflow */
  SOFTMAX_ERR_MISALIGNED = 2,  /* a forced vector/bulk-copy variant got a base or row pitch not 16-B aligned */
  SOFTMAX_ERR_UNSUPPORTED = 3, /* a forced variant cannot take this shape (row too large, ...) */
  SOFTMAX_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  SOFTMAX_ERR_TIMEOUT = 5      /* a kernel's bounded wait ran out (reported by softmax_get_status) */
};

/* Kernel variants (softmax_rows_ex).  AUTO picks one from the shape. */
enum softmax_variant {
  SOFTMAX_VARIANT_AUTO = 0,
  /* One read: the row is loaded once into registers with 128-bit loads (rows up to 64 KiB; AUTO
     takes it for fp32 rows up to 64 KiB and 16-bit rows up to 4 KiB). */
  SOFTMAX_VARIANT_ONEREAD_REG = 1,
  /* One read: bulk copies (cp.async.bulk + mbarrier) stage whole rows in shared memory.  Rows
     up to 8 KiB: each warp owns a row at a time and a private ring of row slots that its lane 0
     refills; longer rows (up to 64 KiB; fp32 rows up to 128 KiB, 16-bit rows up to 120 KiB, kept
     packed): a producer warp feeds a CTA-wide consumer group that copies the row to registers
     and frees the slot at once; longer
     rows (16-byte aligned, up to 1 MiB): a thread-block cluster of 2-8 CTAs per row, each CTA's
     segment held in shared and tensor memory until the row's state, merged over distributed
     shared memory, is known.  AUTO takes the last for many rows of 128 - 512 KiB and 768 KiB - 1 MiB. */
  SOFTMAX_VARIANT_ONEREAD_SMEM = 2,
  /* Two passes over global memory: online fold with 128-bit loads, then re-read and normalise
     (any N; the re-read is served from L2 while the row is still resident).  Aligned rows above
     64 KiB run on the cluster-row kernel: rows of ~260 KiB and more are shared by a thread-block
     cluster (2-16 CTAs, states merged over distributed shared memory), so that the rows in
     flight stay within L2. */
  SOFTMAX_VARIANT_TWOPASS = 3,
  /* Split row: one row is spread over every CTA of the grid; CTAs of a thread-block cluster merge
     (m, d) over distributed shared memory, clusters exchange 8-byte states through global memory
     (16-byte aligned rows above about 150 KiB).  Each CTA holds its segment of a row in shared
     memory from the load until the normalisation, so x is read once: rows up to about 17 MB on
     a 152-SM GB300 (at least two segments per SM fit in shared memory; shorter rows keep up to
     eight in flight).  Longer rows run SOFTMAX_VARIANT_SPLITROW_STREAM instead (and
     softmax_last_variant() reports that).  AUTO takes the split row for rows of 8 MiB and more at
     any row count, and for rows of 4 MiB and more when there are at most 16 of them.
     It needs every cluster resident at once, so it must not share the GPU with other kernels
     (softmax_rows_host never uses it): kernels running beside it on other streams can keep
     clusters off the GPU until the exchange wait runs out (SOFTMAX_ERR_TIMEOUT, y undefined). */
  SOFTMAX_VARIANT_SPLITROW = 4,
  /* Split row, streaming: as SOFTMAX_VARIANT_SPLITROW, but nothing of a row is held on chip, so
     rows of any length are taken: every CTA streams its segment twice through a ring of
     shared-memory slots, the fold, then the normalisation, whose re-read is served from L2 while
     the next rows fold. */
  SOFTMAX_VARIANT_SPLITROW_STREAM = 5
};

/*
 * softmax_rows -- y = softmax(x) along each row ("5.2 CUDA Online Softmax
 * 实现优化", §2.2, the whole method).  x and y: device, M x N, dtype.  y may
 * not overlap x unless y == x (in place).
 */
int softmax_rows(const void* x, void* y, int64_t M, int64_t N, int dtype, void* stream);

/*
 * softmax_rows_ex -- softmax_rows with optional per-row state outputs
 * (m_out, d_out, lse_out: fp32[M] or NULL) and a forced variant.  The state
 * is the (m, d) pair each row's online fold ends with ("5.2 CUDA Online
 * Softmax 实现优化", §2.1; "Softmax 数值稳定性与 IO-Aware Attention" §四, the
 * mergeable state) and LSE = m + ln d ("从原始Softmax到在线Softmax",
 * log-sum-exp); the variants are the page's kernel designs re-made for this
 * GPU: the register one-read kernel of §6, the two passes of §2.2 with the
 * vector loads of §5, and the split rows of §7.1.
 * A forced variant that needs 16-byte alignment returns SOFTMAX_ERR_MISALIGNED
 * when x, y or the row pitch N * sizeof(dtype) is not a multiple of 16;
 * AUTO never does (it falls back to scalar-access kernels).
 */
int softmax_rows_ex(const void* x, void* y, float* m_out, float* d_out, float* lse_out, int64_t M,
                    int64_t N, int dtype, int variant, void* stream);

/*
 * softmax_rows_causal -- softmax_rows_ex for rows masked by position, as in causal attention
 * scores: row r keeps its first
 *     L_r = clamp(r % q_period + 1 + key_offset, 0, N)
 * entries (query q = r % q_period sees keys 0 .. q + key_offset; key_offset = 0 when queries and
 * keys have the same length), and entries j >= L_r count as -inf.  Masked entries are never read
 * -- their bytes may hold anything -- and y is 0 there, so each row reads L_r elements instead of
 * N: the block skipping of FlashAttention-2 ("Softmax 数值稳定性与 IO-Aware Attention" §八,
 * skipping the causal mask's invalid blocks) applied to the plain softmax.  A row with L_r = 0
 * gives y = 0, m = -inf, d = 0, LSE = -inf.  q_period >= 1 (else SOFTMAX_ERR_INVALID_ARG); other
 * arguments as softmax_rows_ex.  Rows of at most 16 KiB (16-byte aligned) run one warp per row
 * loading only the live prefix; other rows run the two-pass kernel over the live prefix.
 */
int softmax_rows_causal(const void* x, void* y, float* m_out, float* d_out, float* lse_out, int64_t M,
                        int64_t N, int64_t q_period, int64_t key_offset, int dtype, void* stream);

/* Flags of softmax_rows_strided. */
enum softmax_flags { SOFTMAX_FLAG_LOG = 1 /* y = log softmax instead of softmax */ };

/*
 * softmax_rows_strided -- softmax_rows_ex with a row pitch, a scale and an output choice:
 *     y[r, j] = softmax(scale * x[r, :])_j        (flags = 0)
 *     y[r, j] = log softmax(scale * x[r, :])_j    (flags = SOFTMAX_FLAG_LOG)
 * for r < M, j < N, where row r of x starts at element r * ldx and row r of y at r * ldy (a
 * column block of a wider matrix, or rows with padding).  The scale folds into the exponent slope
 * (scale * log2 e), as attention's 1/sqrt(d) does, at no cost per element; the state outputs
 * describe scale * x: m_out = scale * max_j x[r, j] (rounded once, the maximum of the rounded
 * products), d_out relative to it, LSE = m_out + ln d.
 *   ldx, ldy -- row pitches in ELEMENTS, >= N (0 means N).
 *   scale    -- finite and > 0 (else SOFTMAX_ERR_INVALID_ARG); 1 gives softmax_rows_ex's result.
 *   flags    -- 0 or SOFTMAX_FLAG_LOG.
 *   variant  -- AUTO, ONEREAD_REG, ONEREAD_SMEM (the CTA bulk-copy kernel; for contiguous rows
 *               at scale 1 beyond its reach, the cluster kernel that holds each row on chip) or
 *               TWOPASS; SPLITROW gives SOFTMAX_ERR_UNSUPPORTED.  The vector and bulk-copy paths also need ldx * s and
 *               ldy * s to be multiples of 16 bytes (a forced ONEREAD_SMEM otherwise returns
 *               SOFTMAX_ERR_MISALIGNED; AUTO takes the scalar paths).
 * x and y may be the same matrix (x == y, ldx == ldy); other overlaps are undefined.  Other
 * arguments and errors as softmax_rows_ex.
 */
int softmax_rows_strided(const void* x, int64_t ldx, void* y, int64_t ldy, float* m_out, float* d_out,
                         float* lse_out, int64_t M, int64_t N, int dtype, float scale, int flags, int variant,
                         void* stream);

/*
 * log_softmax_rows -- y = log softmax(x) row by row: y_j = x_j - LSE with LSE = m + ln d
 * ("从原始Softmax到在线Softmax", section "softmax实际代码实现": log_probs = logits - max -
 * log(sum_exp), the step before the cross-entropy loss).  Computed as (x_j - m) - ln d from the
 * online state, so x is read once as for softmax.  An all -inf row gives y = -inf everywhere
 * (log 0).  Arguments, layout, outputs and errors as softmax_rows_ex; `variant` may be AUTO,
 * ONEREAD_REG, ONEREAD_SMEM (the bulk-copy kernels, and for many rows of 128 - 512 KiB and 768 KiB - 1 MiB a
 * thread-block cluster per row held on chip) or TWOPASS.  SPLITROW gives
 * SOFTMAX_ERR_UNSUPPORTED; AUTO never picks it (a single very long row runs TWOPASS).
 */
int log_softmax_rows(const void* x, void* y, float* m_out, float* d_out, float* lse_out, int64_t M,
                     int64_t N, int dtype, int variant, void* stream);

/*
 * cross_entropy_rows -- per-row cross-entropy loss against integer labels:
 *     loss[r] = LSE_r - x[r, labels[r]]  ( = -log softmax(x_r)[labels[r]] )
 * ("从原始Softmax到在线Softmax", section "softmax实际代码实现", cross_entropy_loss, and the
 * worked example "交叉熵损失计算": logits [2.0, 1.0, 0.1], label 0 -> 0.4170), evaluated as
 * (m - x_label) + ln d in the page's order (no cancellation for large |m|).  The page
 * returns the mean over rows; this call returns each row's loss (the mean is the caller's sum
 * over loss / M).  Only x is read (no y is written): one pass over each row for the online
 * state, plus the labelled element.
 *   labels  -- device, int64, M entries.  A negative label marks a row to ignore: loss = 0.
 *              A label >= N gives loss = NaN, x is not read there, and the next
 *              softmax_get_status() returns SOFTMAX_ERR_INVALID_ARG.
 *   loss    -- device, fp32, M entries (required).
 *   lse_out -- device, fp32, M entries, or NULL.
 * Other arguments and errors as softmax_row_state.
 */
int cross_entropy_rows(const void* x, const int64_t* labels, float* loss, float* lse_out, int64_t M, int64_t N,
                       int dtype, void* stream);

/*
 * attention_forward -- O = softmax(scale Q K^T) V row by row, without forming S = Q K^T in memory:
 * the blocked online recurrence of "从原始Softmax到在线Softmax" (m' = max(m, block max),
 * l = e^(m - m') l + sum e^(s - m'), o~ = e^(m - m') o~ + sum e^(s - m') v, o = o~ / l), the
 * FlashAttention forward tile of "5.2 CUDA Online Softmax 实现优化" §8.2, on the tensor cores.
 *   q       -- device, [BH][Sq][d] row-major, dtype elements.
 *   k, v    -- device, [BH][Sk][d].
 *   o       -- device, [BH][Sq][d] (written).
 *   lse_out -- device, fp32 [BH][Sq]: m + ln l of each row (natural log, of scale Q K^T), or NULL.
 *   scale   -- finite, > 0; 0 means 1/sqrt(d), attention's usual scale (rounded to fp32).
 *   causal  -- 1: query row i sees keys j <= i + Sk - Sq (the last query sees every key); 0: all.
 * A row that sees no key gets o = 0, LSE = -inf.  Supported: dtype SOFTMAX_BF16 or SOFTMAX_F16
 * with d = 64 or 128 (fp32 accumulation; P rounded to the element type for the P V product; fp16
 * weights stay below 2^8, O below max |v|); other dtypes or head sizes return
 * SOFTMAX_ERR_UNSUPPORTED, as do BH > 65535 and Sq or Sk > 2^31 - 256.
 * Pointers 16-byte aligned (else SOFTMAX_ERR_MISALIGNED).
 * BH == 0 is a no-op.  A bounded wait that runs out is reported by softmax_get_status.
 */
int attention_forward(const void* q, const void* k, const void* v, void* o, float* lse_out, int64_t BH, int64_t Sq,
                      int64_t Sk, int64_t d, float scale, int causal, int dtype, void* stream);

/*
 * softmax_row_state -- only the per-row state (m, d) and LSE: the first pass
 * of the online method ("5.2 CUDA Online Softmax 实现优化", §2.2, pass 1;
 * "Softmax 数值稳定性与 IO-Aware Attention" §四, the mergeable state).  Reads x
 * once; writes 12 bytes per row at most.  At least one of m_out, d_out,
 * lse_out must be non-NULL.  With merge_states this lets a caller fold a row
 * in pieces.
 */
int softmax_row_state(const void* x, float* m_out, float* d_out, float* lse_out, int64_t M,
                      int64_t N, int dtype, void* stream);

/*
 * merge_states -- elementwise merge of two arrays of row states
 * ("5.2 CUDA Online Softmax 实现优化", §4.1; "Softmax 数值稳定性与 IO-Aware
 * Attention" §4.1):  m = max(m_a, m_b),  d = d_a e^(m_a - m) + d_b e^(m_b - m),
 * with (-inf, 0) the identity.  Inputs: fp32[M] device arrays (all required).
 * Outputs: fp32[M] device arrays, m_out and d_out required, lse_out optional.
 * Outputs may alias the inputs of the same index (in place).
 */
int merge_states(const float* m_a, const float* d_a, const float* m_b, const float* d_b,
                 float* m_out, float* d_out, float* lse_out, int64_t M, void* stream);

/*
 * softmax_rows_host -- softmax_rows on HOST buffers (x_host, y_host: M x N of
 * dtype).  When both buffers are page-locked (cudaHostAlloc / cudaHostRegister,
 * e.g. torch pin_memory) and rows are at most 32 KiB, the register one-read
 * kernel reads x and writes y in host memory directly over the host link
 * (zero-copy).  Otherwise row blocks of about 8 MiB are copied host->device,
 * normalised in place on the GPU and copied back, with the copies and kernels
 * of consecutive blocks overlapped on three internal streams; those streams and
 * the device staging buffers (3 x one block) are created on the first call on
 * a device and kept until the process exits, and concurrent calls on one
 * device are serialised.  Returns when y_host holds the result (the call
 * synchronises).  `stream` orders the work after earlier work on that stream.
 */
int softmax_rows_host(const void* x_host, void* y_host, int64_t M, int64_t N, int dtype,
                      void* stream);

/*
 * softmax_rows_splitrow_noalloc -- the split-row softmax (SOFTMAX_VARIANT_SPLITROW, with the same
 * choice between the on-chip and the streaming kernel) for callers that cannot allocate device
 * memory.  The pages describe no such call; it exists for callers
 * such as code held to a device-memory budget fixed in advance, code whose framework allocator
 * owns the device memory, or host threads that must not make a call that may block or
 * synchronise the device.  It allocates nothing (no cudaMalloc, cudaMallocAsync, cudaFree or
 * library allocator): the exchange scratch lives in a fixed 320 KiB device array inside the
 * library (40960 slots of 8 bytes), present on every device that loads the library until the
 * process exits.
 *  - Arguments as softmax_rows_ex (device pointers; x, y 16-byte aligned with N * sizeof(dtype)
 *    a multiple of 16, else SOFTMAX_ERR_MISALIGNED).
 *  - Capacity: M x (number of clusters) <= 40960 slots; with the 19 clusters of 8 CTAs used on a
 *    152-SM GB300 that is M <= 2155 rows (at least 512 rows with up to 80 clusters).  Larger M,
 *    or rows the split kernel cannot take, return SOFTMAX_ERR_UNSUPPORTED without launching.
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress, with
 *    that device current) and keeps it; make that first call before any stream capture.
 *  - Like SOFTMAX_VARIANT_SPLITROW it needs every SM of the GPU: kernels running beside it on
 *    other streams can keep its clusters off the GPU until the exchange wait runs out, and the
 *    call then reports SOFTMAX_ERR_TIMEOUT (through softmax_get_status) with y undefined.
 *  - Every call shares the one array and resets the part it uses (a cudaMemsetAsync on `stream`
 *    before the kernel); calls whose executions overlap on the GPU -- on different streams, or
 *    from different threads -- race on it and must be serialised by the caller.
 */
int softmax_rows_splitrow_noalloc(const void* x, void* y, float* m_out, float* d_out, float* lse_out,
                                  int64_t M, int64_t N, int dtype, void* stream);

/*
 * softmax_get_status -- synchronises `stream`, then returns and clears the
 * status word of the current device: SOFTMAX_OK, or the error a kernel
 * recorded since the last call (SOFTMAX_ERR_TIMEOUT for a bounded wait that
 * ran out, which takes precedence; SOFTMAX_ERR_INVALID_ARG for a cross-entropy
 * label >= N).  SOFTMAX_ERR_CUDA if the synchronisation itself failed.
 */
int softmax_get_status(void* stream);

/* A static, human-readable name for a status code. */
const char* softmax_status_string(int status);

/* The CUDA error string of the last SOFTMAX_ERR_CUDA on this host thread ("" if none). */
const char* softmax_last_cuda_error(void);

/* The variant (enum softmax_variant) the last successful compute call on this host thread ran. */
int softmax_last_variant(void);

/*
 * softmax_debug_set_fault -- test hook.  fault = 1 makes the next
 * split-row launches skip one cluster's state publication, so every other
 * cluster's bounded wait runs out and the kernel records SOFTMAX_ERR_TIMEOUT
 * instead of hanging; fault = 2 makes the next attention_forward launches with
 * at most 256 keys (Sk <= 256, two key tiles) skip the copy of the first V
 * tile, with the same outcome (the output is then undefined); longer key
 * sequences ignore it.  fault = 0 restores normal behaviour.  Returns the
 * previous value.  Process-wide; not for production use.
 */
int softmax_debug_set_fault(int fault);

/* The wait limit of the split-row exchange and of every wait in attention_forward, in nanoseconds
 * (default 200 ms).  Returns the old value. */
int64_t softmax_debug_set_wait_limit_ns(int64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* ROW_WISE_ONLINE_SOFTMAX_ROWS_H */
