/*
 * kq.h -- C ABI of the GB300 (sm_103a) K-quant matvec library, libkq.so.
 *
 * The operation ("Chapter 13 - The QKV + gate matvec family", section 13.1):
 *
 *     y[t][i] = sum_{j=0..cols-1} W[i,j] * x[t][j],   i < rows, t < ntok,
 *
 * where W is stored row-major in llama.cpp-style K-quant super-blocks of 256
 * weights and is dequantized on the fly, never written out ("Chapter 6 - The
 * kquant family on the reference lane", sections 6.2 and 6.4):
 *
 *     Q4_K  144 B / block   w = d*sc_j*nibble - dmin*m_j        (Figure 6.2)
 *     Q5_K  176 B / block   w = d*sc_j*(nibble | hbit<<4) - dmin*m_j  (6.4)
 *     Q6_K  210 B / block   w = d*sc_j*(code - 32), 16 int8 scales   (6.5)
 *
 * x and y are f32.  A matrix is computed with one of two arithmetics,
 * chosen from its format, cols and ntok alone:
 *   - integer (dp4a) block sums, for 1 token column, and for 2..3 unless
 *     ntok x (cols / 256) x the record bytes (832 for Q4_K / Q5_K, 1056
 *     for Q6_K) passes 140 KB;
 *   - the tensor cores (mma.sync m16n8k16, f16 operands, f32 accumulation;
 *     "Chapter 6", section 6.8, the weight-stationary tile for many
 *     columns) otherwise, i.e. for 4..16 token columns and for wide
 *     matrices at 2..3: a short pass turns x into f16 operand fragments,
 *     then one launch reads W once for all the columns.
 * A token column's result depends on its own inputs and on the arithmetic
 * -- never on the other columns, the number of rows or the other members
 * of a set (a set that mixes the two runs one launch per arithmetic).
 *
 * Conventions for every entry point below
 *   - W is a DEVICE pointer (cudaMalloc / torch CUDA storage on the current
 *     device).  x and y are device pointers too, or pointers into pinned
 *     host memory (cudaHostAlloc, cudaHostRegister, torch pin_memory).  A
 *     host y is written in place by the kernel over the host link.  Host
 *     x planes are copied once into a stream-ordered device temporary by a
 *     small staging kernel, which the matvec overlaps with its weight
 *     stream (kq_matvec_noalloc instead reads them in place).  On GB300
 *     (Grace) this replaces the separate copies in and out.  Managed memory
 *     is accepted for x and y.  Anything else (pageable host memory,
 *     another device's memory) is KQ_ERR_MEMORY.  All memory is owned by
 *     the caller.  The library
 *     keeps no pointer after a call returns and never synchronizes.  Its
 *     allocations are stream-ordered temporaries (cudaMallocAsync /
 *     cudaFreeAsync on `stream`): the input records of calls whose records
 *     do not fit in shared memory, the fragments of the tensor-core
 *     arithmetic (8704 bytes per 256 inputs per group of 8 columns), and
 *     staged host inputs; kq_matvec_set_ws takes them from a caller's
 *     workspace instead, and kq_matvec_noalloc allocates nothing.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *     the legacy default stream) and may be captured in a CUDA graph.
 *   - Every argument is validated on the host before anything is launched;
 *     a call that returns an error has enqueued nothing, with one exception:
 *     KQ_ERR_CUDA from a later launch of a call that runs as several (the
 *     staging, fragment or record pass and the matvec), after the earlier
 *     ones had been enqueued.  KQ_ERR_CUDA means a launch itself failed;
 *     kq_last_cuda_error() returns the CUDA error code of the most recent
 *     such failure on the calling thread.
 *   - Results are deterministic: a row's arithmetic depends only on the
 *     format, cols, ntok and that row's bytes and inputs -- not on the grid,
 *     the number of rows, or which other matrices share the launch.
 *   - Accuracy and its precondition.  Products are summed exactly in
 *     integers over inputs held in 24-bit fixed point, one power-of-two step
 *     per group of 32 consecutive inputs set by the group's largest
 *     magnitude (2^(E-1) <= max|x| < 2^E, E clamped to [-100, 128]).  The
 *     input rounding adds at most  B_i = sum_g 2^(E_g - 24) * sum_{j in g}
 *     |W_ij|  to output i's error; the sub-block sums add f32 roundings
 *     far smaller.  The result is within |y - y_exact| <= 1e-4 * S_i +
 *     1e-6, S_i = sum_j |W_ij x_j|, whenever B_i is below that bound:
 *     PRECONDITION, in words: no input is more than about 10^4 times the
 *     typical magnitude of its group of 32 while sitting on a (near) zero
 *     weight.  Inputs drawn from one distribution (as activations are) are
 *     hundreds of times inside it; an input of 1e6 on an exactly zero
 *     weight among N(0,1) inputs is about 10x outside it, though still
 *     within B.  NaN or infinite inputs make the outputs that read their
 *     group NaN.  This holds for the dp4a arithmetic.
 *     The tensor-core arithmetic holds each input as two f16
 *     terms after scaling its 256-input column by a power of two: an input
 *     error of at most max(2^-22 |x_j|, 2^(E-39)), max|x| < 2^E over the
 *     column; codes times these terms are exact and the sums are f32.  The
 *     same contract holds there with the precondition relaxed to inputs up
 *     to about 10^7 times their column's typical magnitude on a zero
 *     weight.  On both paths a row whose weights are all exactly zero gives
 *     exactly zero.  NaN or infinite inputs make the outputs that read their
 *     256-input column NaN.
 */
#ifndef KQ_H
#define KQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Format codes: the GgmlType values of the three K-quant formats
 * ("Chapter 6 - The kquant family on the reference lane", section 6.1). */
typedef enum kq_fmt {
    KQ_Q4_K = 12,
    KQ_Q5_K = 13,
    KQ_Q6_K = 14
} kq_fmt;

typedef enum kq_status {
    KQ_OK = 0,
    KQ_ERR_FORMAT = 1,  /* fmt is not one of kq_fmt                          */
    KQ_ERR_SHAPE = 2,   /* rows < 1, cols < 256, cols % 256 != 0, or too big  */
    KQ_ERR_NTOK = 3,    /* ntok outside 1..KQ_MAX_NTOK                        */
    KQ_ERR_NULL = 4,    /* a required pointer is NULL                         */
    KQ_ERR_ALIGN = 5,   /* W or x not 16-byte aligned, or y not 4-byte aligned */
    KQ_ERR_ALIAS = 6,   /* an output overlaps an input or another output      */
    KQ_ERR_CUDA = 7,    /* a CUDA call failed (see kq_last_cuda_error)        */
    KQ_ERR_TIMEOUT = 8, /* a bounded device-side wait expired                 */
    /* codes beyond the eight of the problem statement's boundary:          */
    KQ_ERR_COUNT = 9,   /* set size outside 1..KQ_MAX_SET                     */
    KQ_ERR_LIMIT = 10,  /* a fixed buffer too small: kq_matvec_noalloc's, or a
                           kq_matvec_set_ws workspace                         */
    KQ_ERR_MEMORY = 11  /* W not in this device's memory, or x / y in memory
                           the device cannot address (pageable host memory,
                           another device's memory)                        */
} kq_status;

#define KQ_MAX_NTOK 16
#define KQ_MAX_SET 16
/* Largest accepted cols (inputs per row). */
#define KQ_MAX_COLS (1LL << 20)
/* Largest accepted rows per matrix. */
#define KQ_MAX_ROWS (1LL << 30)

/*
 * Bytes per 256-weight super-block of `fmt` (144, 176 or 210; Figure 6.1 of
 * "Chapter 6 - The kquant family on the reference lane"), or -1 if `fmt` is
 * not a kq_fmt.  Pure host function.
 */
int64_t kq_block_bytes(int fmt);

/*
 * Bytes of a rows x cols matrix of `fmt`: rows * (cols/256) * block bytes,
 * rows stored one after another with no padding (section 6.6 of the same
 * chapter).  -1 if fmt, rows or cols is invalid.  Pure host function.
 */
int64_t kq_matrix_bytes(int fmt, int64_t rows, int64_t cols);

/*
 * One K-quant matvec ("Chapter 13 - The QKV + gate matvec family", sections
 * 13.1 and 13.4; "Chapter 6", section 6.7).
 *
 *   fmt   kq_fmt of W.
 *   W     device pointer, kq_matrix_bytes(fmt, rows, cols) bytes, row-major
 *         super-blocks; 16-byte aligned.  Read only.
 *   rows  output rows, 1..KQ_MAX_ROWS.
 *   cols  inputs per row, a positive multiple of 256, at most KQ_MAX_COLS.
 *   x     device or pinned host pointer, f32 [ntok][cols], contiguous,
 *         16-byte aligned.  Read only.
 *   y     device or pinned host pointer, f32 [ntok][rows], contiguous,
 *         4-byte aligned.  Overwritten (not accumulated).  Must not overlap
 *         W or x.
 *   ntok  token columns, 1..KQ_MAX_NTOK.
 *   stream  cudaStream_t or NULL.
 *
 * Returns KQ_OK after enqueueing its kernel(s), or an error code (see the
 * conventions above).  The pointers are checked with cudaPointerGetAttributes
 * (KQ_ERR_MEMORY) after the host-only checks.
 */
kq_status kq_matvec(int fmt, const void *W, int64_t rows, int64_t cols,
                    const float *x, float *y, int ntok, void *stream);

/*
 * One member of a matvec set: a matrix, the input it reads and the output
 * it writes.  Fields have the meaning and rules of kq_matvec's arguments.
 */
typedef struct kq_mat {
    int32_t fmt;
    int32_t reserved;   /* must be 0 */
    const void *W;
    int64_t rows;
    int64_t cols;
    const float *x;
    float *y;
} kq_mat;

/*
 * Several independent matvecs in ONE kernel launch, the grid split among
 * them -- the "concurrent set" of four projections that share one read-only
 * input and write disjoint outputs ("Chapter 13 - The QKV + gate matvec
 * family", section 13.5), and the grid-split pair of two matrices of
 * possibly different formats, each with its own input plane (audit note
 * "opus_gdn_qsa", section 1, gemv_cat).
 *
 *   mats   host array of n kq_mat descriptors (read during the call only).
 *   n      1..KQ_MAX_SET.
 *   ntok   token columns shared by all members, 1..KQ_MAX_NTOK.
 *   stream cudaStream_t or NULL.
 *
 * Members may differ in fmt, rows and cols; they may share x (and even W).
 * Each y must not overlap any W, any x, or another member's y.  Each
 * member's y is bitwise identical to what kq_matvec would write for it.
 * Returns as kq_matvec; on error nothing is enqueued for any member.
 */
kq_status kq_matvec_set(const kq_mat *mats, int n, int ntok, void *stream);

/*
 * Device workspace bytes that kq_matvec_set_ws needs for this set and ntok:
 * room for every member's x as if it were staged, the tensor-core
 * fragments of the members computed on the tensor cores, and the dp4a input
 * records of the largest token chunk.  An upper bound of what the call
 * uses, from the shapes and formats alone (no pointer is read or queried;
 * no GPU is touched).  A negative kq_status for a set kq_matvec_set would
 * reject on its arguments alone.
 */
int64_t kq_workspace_bytes(const kq_mat *mats, int n, int ntok);

/*
 * kq_matvec_set with a caller-provided device workspace instead of the
 * library's stream-ordered temporaries: the call allocates nothing, so the
 * work it enqueues is kernels only.  With launch overlap on
 * (kq_set_overlap), in a CUDA graph or a stream, the tensor-core fragment
 * pass can then start while the kernel before it still runs, where an
 * allocation between the kernels would have made it wait for that kernel
 * to finish and launch afterwards.  The library launches it that way
 * before a direct-load launch and before a streaming launch whose CTAs
 * keep all their weight stages in flight at once, where it was measured
 * faster.
 *
 *   ws        device (or managed) memory of the current device, 256-byte
 *             aligned, not overlapping any member's W, x or y.  Owned by the
 *             caller; the call's work on `stream` uses it until it has
 *             finished, so calls that may run at the same time (different
 *             streams, or graphs replayed concurrently) need separate
 *             workspaces.  Its contents need not be initialised and are
 *             garbage afterwards.
 *   ws_bytes  at least kq_workspace_bytes(mats, n, ntok).
 *
 * Results are bitwise those of kq_matvec_set.  Errors as kq_matvec_set,
 * plus, with nothing enqueued: KQ_ERR_LIMIT (ws_bytes too small),
 * KQ_ERR_NULL (ws NULL), KQ_ERR_ALIGN (ws not 256-byte aligned),
 * KQ_ERR_ALIAS (ws overlaps a member's buffers), KQ_ERR_MEMORY (ws not
 * this device's memory).
 */
kq_status kq_matvec_set_ws(const kq_mat *mats, int n, int ntok, void *stream, void *ws,
                           int64_t ws_bytes);

/*
 * Rows of a K-quant matrix gathered by index and dequantized to f32 -- the
 * embedding lookup ("Chapter 6 - The kquant family on the reference lane",
 * section 6.7, muser_embedding_q4k: the token's row of the Q4_K embedding
 * table, dequantized element by element with section 6.3's formula), for
 * any of the three formats:
 *
 *   out[i][j] = W[ids[i], j],  i < n, j < cols
 *
 *   fmt, W, rows, cols  as kq_matvec (W device, 16-byte aligned).
 *   ids   device or pinned host int32[n], 4-byte aligned; an index outside
 *         [0, rows) yields a row of NaN.
 *   n     rows to gather, 0..2^31-1 (0: nothing is enqueued).
 *   out   device or pinned host f32 [n][cols], 16-byte aligned,
 *         overwritten; must not overlap W or ids.
 *
 * Each value is the correctly rounded weight: d*sc*q - dmin*m (Q4_K,
 * Q5_K) or d*sc*(q-32) (Q6_K) with only the final subtraction rounded
 * (the products are exact in f32), so any exact evaluation gives the same
 * bits.  Validation and status codes as kq_matvec: after the host-only
 * checks the three pointers are checked with cudaPointerGetAttributes, and
 * W outside this device's memory, or ids / out in memory the device cannot
 * address (pageable host memory, another device's memory), return
 * KQ_ERR_MEMORY with nothing enqueued.  Allocates nothing.
 */
kq_status kq_dequant_rows(int fmt, const void *W, int64_t rows, int64_t cols,
                          const int32_t *ids, int64_t n, float *out, void *stream);

/* Static English text for a status code (never NULL). */
const char *kq_status_str(int status);

/* CUDA error code (cudaError_t value) of the calling thread's most recent
 * KQ_ERR_CUDA, or 0. */
int kq_last_cuda_error(void);

/*
 * Device-side failure report.  The kernels bound every wait on a shared-
 * memory barrier by wall time; a wait that expires sets a per-device error
 * word (and the affected outputs to NaN) instead of hanging.  This call
 * SYNCHRONOUSLY reads the word of the current device (a blocking device-to-
 * host copy; it waits for work already submitted that the copy depends on)
 * and returns KQ_ERR_TIMEOUT if it is set, KQ_OK if not.  With clear != 0 a
 * set word is reset.  KQ_ERR_CUDA if the copy fails.
 */
kq_status kq_device_error(int clear);

/*
 * Kernel selection, for testing and measurement: 0 = automatic (the
 * TMA-streaming kernel whenever the shapes can be staged in shared memory,
 * else the direct-load kernel; with 9..16 token columns on the tensor
 * cores, also the direct-load kernel where the streaming kernel's CTAs
 * would hold several row groups that fill less than four fifths of their
 * 16-row tiles), 1 = always the direct-load kernel, 2 = only
 * the streaming kernel (calls it cannot stage return KQ_ERR_SHAPE with
 * nothing enqueued).  Both kernels compute every output with the same
 * arithmetic in the same order, so results do not depend on this setting.
 * Process-wide; the environment variable KQ_KERNEL=direct|stream sets the
 * initial value.  Returns the previous setting; an argument outside 0..2
 * only queries.
 */
int kq_select_kernel(int which);

/*
 * Launch overlap (off by default).  When on, each streaming-kernel launch
 * may begin while the kernel before it on the same stream is still running
 * (programmatic dependent launch): its CTAs start streaming W into shared
 * memory as soon as SMs free up, and wait for the preceding kernel to
 * complete -- with its memory visible -- before they read x or write y.
 * PRECONDITION while on: no W of a call is written by the kernel that
 * immediately precedes the call on its stream (weights that stay constant,
 * as in inference).  Results are unchanged.  Process-wide; returns the
 * previous setting (0/1); an argument other than 0 or 1 only queries.
 */
int kq_set_overlap(int enable);

/*
 * Kernels the calling thread's most recent successful kq_matvec /
 * kq_matvec_set / kq_matvec_noalloc call enqueued, as bits: 1 = the direct-load kernel, 2 = the
 * TMA-streaming kernel, 4 = the pass that writes input records to global
 * memory first (when they do not fit in shared memory), 8 = the tensor-core
 * arithmetic (after its fragment pass).
 * 0 before any call.
 */
int kq_last_kernels(void);

/*
 * Number of kernel launches the calling thread's most recent successful
 * kq_matvec / kq_matvec_set / kq_matvec_noalloc call enqueued (the record
 * pass counts as one; a call that runs as several launches counts them
 * all).
 * 0 before any call.
 */
int kq_last_launch_count(void);

/*
 * kq_matvec without any memory allocation.  The pages have no counterpart:
 * this is a library service for callers that must not allocate device
 * memory during the call -- code running under a caller-managed memory
 * budget or allocator that forbids hidden allocations, hot loops that must
 * not take the allocator's locks or latency, and devices or processes where
 * stream-ordered allocation (cudaMallocAsync) is unavailable.
 *
 * Same arguments, result and errors as kq_matvec, computed by the direct-
 * load kernel with its input records (see the record pass) in one fixed
 * file-scope device buffer of KQ_NOALLOC_RECORD_BYTES bytes instead of a
 * stream-ordered temporary.  Calls whose records need more return
 * KQ_ERR_LIMIT with nothing enqueued: with the dp4a arithmetic,
 * ntok * (cols / 256) * 832 bytes for Q4_K / Q5_K, * 1056 bytes for Q6_K;
 * with the tensor cores, ceil(ntok / 8) * (cols / 256) * 8704 bytes of
 * fragments, rounded up to 256 bytes.
 * The records are written in full before they are read, so nothing in the
 * buffer has to start at zero.
 *
 * The first call on a device looks the buffer up (cudaGetSymbolAddress,
 * once per device); make that first call before any stream capture.  Every
 * call shares the one buffer: calls that may overlap on the GPU (different
 * streams, or different host threads without ordering) race and must be
 * serialised by the caller.  Results are bitwise those of kq_matvec with
 * the direct-load kernel.
 */
#define KQ_NOALLOC_RECORD_BYTES (1LL << 20)
kq_status kq_matvec_noalloc(int fmt, const void *W, int64_t rows, int64_t cols,
                            const float *x, float *y, int ntok, void *stream);

/* Library ABI version: (major << 16) | minor. */
int kq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KQ_H */
