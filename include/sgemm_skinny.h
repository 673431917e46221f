/*
 * sgemm_skinny.h -- C ABI of the GB300 (sm_103a) BF16 skinny GEMM library.
 *
 *     y[M,N] = x[M,K] . W[N,K]^T        1 <= M <= 8, BF16 in, FP32 accumulate, BF16 out
 *
 * The operation is the F.linear projection of a decode step with M tokens, as
 * used for the unquantized attention, shared-expert and LM-head projections in
 * vLLM PR #62949 ("SM121 skinny-GEMM plans for the GLM-5.3-Flash BF16 decode
 * projections", Overview and Validation table) and vLLM PR #65306 ("Add SM90
 * skinny GEMM plans for the BF16 decode projections", Overview).  Each weight
 * is read exactly once per call, so the call is bound by HBM bandwidth.
 * M = 1..4 are the decode widths the pages plan for; M = 5..8 cover wider
 * batches (speculative verification), which PR #62949 (Validation, below its
 * cold-L2 table) measured at M = 8 within 2% of cuBLAS and left off its plans.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Element type: raw BF16 bit patterns (sgemm_bf16_t).  Products are formed
 *   exactly and accumulated in FP32; each output is rounded once to BF16,
 *   round-to-nearest-even.  The accumulation order depends only on (N, K) and
 *   the plan, never on M or on the data, so a call is deterministic: the same
 *   inputs and plan give bitwise-identical outputs, and row m of an M-row call
 *   equals the 1-row call on x[m,:] under the same plan.
 * - Layout: x is row-major [M,K] with row stride ldx elements (ldx >= K; the
 *   plain call uses ldx = K); W is row-major [N,K], contiguous (the F.linear
 *   weight layout); y is row-major [M,N] with row stride ldy (>= N).
 * - Memory: every array pointer is a DEVICE pointer on the calling thread's
 *   current CUDA device, owned by the caller.  The library keeps no pointer
 *   after a call returns, so weights may be refreshed in place between calls
 *   or between CUDA-graph replays (the in-place refresh rule of vLLM PR #57617,
 *   "Batch paired KDA gate projections (f_b_proj/g_b_proj) into one bmm",
 *   Purpose and source).
 * - Alignment: x and W must be 16-byte aligned, K a multiple of 8 and ldx a
 *   multiple of 8, so that every row of x and W starts on a 16-byte boundary
 *   (they are read with 128-bit loads).  y is written element by element and
 *   needs only 2-byte alignment; ldy may be any value >= N.
 * - Streams: work is enqueued asynchronously on `stream` (NULL = the legacy
 *   default stream); nothing blocks the host.  A call neither allocates nor
 *   synchronizes unless it needs split-K scratch that does not exist yet (see
 *   sgemm_init), so it can be captured into a CUDA graph.
 * - Errors: arguments are checked on the host before anything is enqueued;
 *   a bad argument returns a status and launches nothing.  There is no CPU
 *   fallback and no fallback to another GEMM library.  A failed launch
 *   returns SGEMM_ERR_CUDA (the CUDA error is left for cudaGetLastError).
 * - Devices: only compute capability 10.3 (GB300, sm_103) is accepted.
 */
#ifndef SGEMM_SKINNY_H
#define SGEMM_SKINNY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Raw BF16 bits: sign(1) | exponent(8) | fraction(7). */
typedef uint16_t sgemm_bf16_t;

/* Identical to cudaStream_t / CUstream; declared here so that this header
 * needs no CUDA header. */
typedef struct CUstream_st *sgemm_stream_t;

typedef enum {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_ARG = 1,        /* null pointer, M outside 1..8, N or K < 1, bad ld, batch */
    SGEMM_ERR_UNSUPPORTED_SHAPE = 2,  /* K not a multiple of 8, or a plan that cannot run it */
    SGEMM_ERR_MISALIGNED = 3,         /* x or W not 16-byte aligned, ldx % 8 != 0, y odd */
    SGEMM_ERR_UNSUPPORTED_DEVICE = 4, /* current device is not compute capability 10.3 */
    SGEMM_ERR_NO_WORKSPACE = 5,       /* split-K scratch missing while the stream is capturing */
    SGEMM_ERR_CUDA = 6                /* a CUDA runtime call or launch failed */
} sgemm_status_t;

/* One launch configuration ("plan") of the kernel.  The fields are the tuning
 * knobs of the skinny-GEMM plan tables in vLLM PR #62949 (Details: block_size,
 * outputs_per_block, k_unroll, vector_width) extended with a split-K factor and
 * a pipeline depth. */
typedef struct {
    int variant;          /* kernel family, see SGEMM_VARIANT_* */
    int threads;          /* threads per CTA (a multiple of 32) */
    int rows_per_warp;    /* output rows n a warp accumulates at once */
    int lanes_per_row;    /* lanes sharing one row: 32, 16 or 8 (16/8 suit small K) */
    int k_unroll;         /* 16-byte W loads per row per lane kept in flight */
    int vec_bytes;        /* bytes per W load: 16 */
    int split_k;          /* K split across this many CTAs (1 = none) */
    int stages;           /* pipeline depth: batches of loads in flight per warp, 1 or 2
                             (2 = double-buffered batches; 0 is read as 1) */
    int ctas_per_sm;      /* resident CTAs per SM the grid is sized for (0 = occupancy max) */
    int id;               /* index in the compiled plan table, or -1 for a heuristic plan */
} sgemm_plan_t;

enum {
    SGEMM_VARIANT_LDG = 0,        /* W streamed with 128-bit non-allocating loads into a ring of
                                     registers, x staged in shared memory, BF16 widened to FP32,
                                     FP32 FMA, warp-shuffle reduction */
    SGEMM_VARIANT_LDG_MIXFMA = 1, /* the same with the mixed-precision FMA (BF16 operands, FP32
                                     addend): fewer instructions, bitwise-identical results */
    SGEMM_VARIANT_MMA = 2,        /* W streamed the same way into mma.sync m16n8k16 tensor-core
                                     fragments (x padded to 8 columns); a CTA of NW warps splits
                                     each 16-row tile's K range and adds the NW partial tiles in
                                     shared memory.  rows_per_warp = 16, lanes_per_row = 4,
                                     k_unroll = 32-element k-blocks per batch */
    /* 3: retired (x as the A operand of mma.sync with CTA-wide 8-row tiles; after the
       tcgen05 kernel arrived it won no cell of the sweep); plans with variant 3 are
       refused with SGEMM_ERR_UNSUPPORTED_SHAPE */
    /* 4: retired (a bulk-copy kernel that no sweep ever selected); plans with
       variant 4 are refused with SGEMM_ERR_UNSUPPORTED_SHAPE */
    SGEMM_VARIANT_LDG_FFMA2 = 5,  /* the streaming kernel of variant 0 with packed FP32x2 FMA
                                     (two partial sums per output, even and odd k, added at the
                                     end): half the FMA instructions */
    SGEMM_VARIANT_LDGX_MIXFMA = 6, /* variant 1 reading x from global memory through L1 at each
                                     use instead of staging it in shared memory (no CTA barrier
                                     before the first FMA); same results as variants 0/1 */
    SGEMM_VARIANT_LDGX_FFMA2 = 7, /* variant 5 with x read the same way; same results as 5 */
    /* 8: retired (the math of variant 3 with warp-owned tiles; it won no cell of the
       sweep); plans with variant 8 are refused with SGEMM_ERR_UNSUPPORTED_SHAPE */
    SGEMM_VARIANT_LDG_MMA = 9,    /* the streaming kernel of variant 1 (one row's 512 bytes per
                                     load instruction, lanes_per_row = 32) with the products
                                     done by mma.sync m16n8k16: the 8 columns of B are the 8
                                     consecutive 32-element segments a warp load covers, A holds
                                     x rows m and m+1 at the same k, and the diagonal of D is the
                                     per-segment dot product (2 MMAs per 16 bytes of W and pair
                                     of x rows, instead of 8 FMAs per x row) */
    SGEMM_VARIANT_TC05 = 10,      /* the Blackwell tensor-core data path: a producer thread streams
                                     boxes of 128 rows x 64 elements of W (and the matching box
                                     of x) with TMA (cp.async.bulk.tensor) into a ring of shared-
                                     memory stages; one thread issues tcgen05.mma (128 rows of W x
                                     16 columns of x, FP32 accumulator in tensor memory); four
                                     warps read the accumulator back and write y.  No W element
                                     passes through registers.  threads = 192, rows_per_warp =
                                     128 (rows per tile), lanes_per_row = 0, k_unroll = boxes
                                     per stage (1..4), stages = ring slots (2..16).
                                     split_k = 1: a persistent grid of ctas_per_sm CTAs per SM
                                     (0 = occupancy) over the tiles; split_k = 2..16: the split_k
                                     CTAs of a thread-block cluster share a tile's K range (in
                                     whole 64-element boxes; ceil(ceil(K/64) / ceil(ceil(K/64) /
                                     split_k)) ranges are used) and add their partial sums in
                                     rank order through distributed shared memory: one launch,
                                     no scratch memory */
    SGEMM_VARIANT_LDG_CLUSTER = 11 /* the kernels of variant 1 with a one-launch split: the split_k
                                     (2..8) CTAs of a row range form a thread-block cluster; rank
                                     0 takes the others' FP32 partial sums into its shared memory
                                     (st.async counted on an mbarrier, a bounded wait) and adds
                                     them in split order from 0, as the second pass adds, so the
                                     bits equal variant 1 with the same split.  No scratch memory,
                                     no second kernel.  Its grid gives each warp one row group at
                                     most (ctas_per_sm is not used); split_k = 1 is variant 1 */
};

/* Launch flags (bit set) for the _ex calls.
 * SGEMM_FLAG_PDL: launch as a programmatic dependent of the previous kernel on
 *   the stream.  The kernel lets the next kernel launch early and waits for
 *   the previous kernel to finish (and its writes to be visible) before it
 *   reads x or writes y, so the results are those of a plain launch; the gain
 *   is that launch latency and the kernel's start-up overlap the previous
 *   kernel's tail.
 * SGEMM_FLAG_WEIGHTS_READONLY (with SGEMM_FLAG_PDL): the caller promises that
 *   W is not written by any work that may still be running on the stream when
 *   this call is reached (for example decode weights that no kernel of the
 *   step modifies).  The kernel then starts streaming W before the previous
 *   kernel finishes. */
#define SGEMM_FLAG_PDL 1u
#define SGEMM_FLAG_WEIGHTS_READONLY 2u
/* TEST ONLY: the kernels that wait on mbarriers make those waits run out
 * (about 0.2 s each) without any fault: the tcgen05 kernel
 * (SGEMM_VARIANT_TC05) issues no copies, and in a cluster-split streaming plan
 * (SGEMM_VARIANT_LDG_CLUSTER, split_k > 1) ranks 1.. send rank 0 no partial
 * sums.  The kernel then writes NaN outputs, sets the device error word and
 * returns.  Exercises failure detection.  Other variants ignore the flag. */
#define SGEMM_FLAG_TEST_STALL 4u

/* y = x . W^T for contiguous x [M,K] and y [M,N].  Plan: sgemm_plan_select(N, K, M). */
sgemm_status_t sgemm_bf16_skinny(const sgemm_bf16_t *x, const sgemm_bf16_t *W, sgemm_bf16_t *y,
                                 int M, int N, int K, sgemm_stream_t stream);

/* As sgemm_bf16_skinny with row strides for x and y, an optional plan
 * (NULL = sgemm_plan_select) and launch flags (SGEMM_FLAG_*; 0 = a plain
 * launch).  A plan that does not fit the shape, or unknown flag bits, return
 * SGEMM_ERR_UNSUPPORTED_SHAPE / SGEMM_ERR_INVALID_ARG; a plan with
 * split_k > 1 needs scratch (sgemm_init). */
sgemm_status_t sgemm_bf16_skinny_ex(const sgemm_bf16_t *x, long long ldx, const sgemm_bf16_t *W,
                                    sgemm_bf16_t *y, long long ldy, int M, int N, int K,
                                    const sgemm_plan_t *plan, unsigned flags,
                                    sgemm_stream_t stream);

/* One independent problem of a batched call.  ldx / ldy are row strides in
 * elements, so x may be a strided view (vLLM PR #57617, Controlled follow-up:
 * the paired inputs are a narrow -> unflatten -> transpose view). */
typedef struct {
    const sgemm_bf16_t *x;
    const sgemm_bf16_t *W;
    sgemm_bf16_t *y;
    long long ldx;
    long long ldy;
} sgemm_pair_t;

#define SGEMM_MAX_BATCH 8

/* `batch` (1..SGEMM_MAX_BATCH) independent GEMMs of one shape (M, N, K) in ONE
 * kernel launch: y_i = x_i . W_i^T.  This is the paired f_b_proj / g_b_proj
 * projection of vLLM PR #57617 (Purpose and source; Microbenchmark table: two
 * launches become one).  `items` is HOST memory, read during the call only
 * (its contents travel as kernel parameters, so the call is graph-capturable).
 * Each item's outputs are bitwise equal to a separate sgemm_bf16_skinny_ex call
 * with the same plan. */
sgemm_status_t sgemm_bf16_skinny_batched(const sgemm_pair_t *items, int batch, int M, int N, int K,
                                         sgemm_stream_t stream);

/* Same, with an explicit plan (NULL = sgemm_plan_select(N, K, M)) and launch
 * flags (SGEMM_FLAG_*, as for sgemm_bf16_skinny_ex). */
sgemm_status_t sgemm_bf16_skinny_batched_ex(const sgemm_pair_t *items, int batch, int M, int N,
                                            int K, const sgemm_plan_t *plan, unsigned flags,
                                            sgemm_stream_t stream);

/* The plan used for (N, K, M): the entry of the compiled sm_103 plan table
 * (filled by the offline sweep under CUDA-graph replay with cold L2, as in
 * vLLM PR #62949, Details, and PR #65306, Details) when it holds one, else a
 * heuristic plan (id = -1).  Pure host function; never fails (arguments out
 * of range give the heuristic plan). */
sgemm_plan_t sgemm_plan_select(int N, int K, int M);

/* Enumerate the compiled kernel configurations (for sweeps and tests):
 * sgemm_plan_count() of them, index 0..count-1; split_k and ctas_per_sm of a
 * returned plan may be changed freely before use.  Returns SGEMM_ERR_INVALID_ARG
 * for an index out of range. */
int sgemm_plan_count(void);
sgemm_status_t sgemm_plan_get(int index, sgemm_plan_t *plan);

/* Whether `plan` can run (M, N, K): SGEMM_OK or the status a call would return. */
sgemm_status_t sgemm_plan_check(const sgemm_plan_t *plan, int M, int N, int K);

/* Allocate the split-K scratch for the current device (idempotent; about
 * 16 MiB of device memory, kept until process exit).  Calls with a split-K
 * plan do this themselves on first use, but a first use inside stream capture
 * cannot allocate and returns SGEMM_ERR_NO_WORKSPACE: call sgemm_init (or run
 * one call eagerly) before capturing.  Split-K calls on one device share this
 * scratch, so split-K calls that may run at the same time on different
 * streams must be ordered by the caller. */
sgemm_status_t sgemm_init(void);

/* One GEMM of a decode chain with that elementwise step fused into its
 * epilogue: y = x . W^T as sgemm_bf16_skinny_ex (same plan, same bits), and
 *     x_next[m][k] = RNE_bf16( float(y[m][k mod N]) * scale )  for 0 <= k < n_next
 * from the BF16 value just stored, so x_next is bitwise what
 * sgemm_bf16_rescale would make from y (vLLM PR #65306, Validation, and its
 * decode-chain protocol: one GEMM per projection, the next input formed from
 * the previous output).  Saves one kernel launch per GEMM of the chain.
 * - x_next: DEVICE array, row stride ld_next >= n_next elements, 2-byte aligned,
 *   overlapping none of x, W and y (else SGEMM_ERR_INVALID_ARG; the kernel
 *   still reads x and W while it writes x_next).  1 <= n_next < 2^31.
 * - With SGEMM_FLAG_PDL the next GEMM on the stream waits for this one before it
 *   reads x_next, as for y.  Other arguments and errors as sgemm_bf16_skinny_ex. */
sgemm_status_t sgemm_bf16_skinny_rescale_ex(const sgemm_bf16_t *x, long long ldx,
                                            const sgemm_bf16_t *W, sgemm_bf16_t *y, long long ldy,
                                            int M, int N, int K, sgemm_bf16_t *x_next,
                                            long long ld_next, long long n_next, float scale,
                                            const sgemm_plan_t *plan, unsigned flags,
                                            sgemm_stream_t stream);

/* y = x . W^T with FP32 outputs: the FP32 sums are stored without rounding to
 * BF16.  For projections whose consumer wants FP32, such as the MoE router gate
 * (288, 4096) that vLLM PR #62949 (Validation, the nsys census) leaves on cuBLAS
 * because of its FP32 output.  Same kernels, plans and accumulation order as
 * sgemm_bf16_skinny_ex; y is a DEVICE array of float, row stride ldy >= N
 * elements, 4-byte aligned (else SGEMM_ERR_MISALIGNED).  Other arguments and
 * errors as sgemm_bf16_skinny_ex. */
sgemm_status_t sgemm_bf16_skinny_f32out_ex(const sgemm_bf16_t *x, long long ldx,
                                           const sgemm_bf16_t *W, float *y, long long ldy, int M,
                                           int N, int K, const sgemm_plan_t *plan, unsigned flags,
                                           sgemm_stream_t stream);

/* The elementwise step between consecutive GEMMs of a decode chain (vLLM PR
 * #65306, Validation: the chain's GEMMs are separated by a short elementwise
 * kernel):
 *     x[k] = RNE_bf16( float(y[k mod n_src]) * scale )   for 0 <= k < n_dst.
 * y and x are DEVICE arrays of BF16 bits (2-byte aligned, not overlapping).
 * flags: SGEMM_FLAG_PDL launches it as a programmatic dependent (it waits for
 * the previous kernel before reading y).  Errors as for the GEMM calls. */
sgemm_status_t sgemm_bf16_rescale(const sgemm_bf16_t *y, long long n_src, sgemm_bf16_t *x,
                                  long long n_dst, float scale, unsigned flags,
                                  sgemm_stream_t stream);

/* Size of the fixed device array used by sgemm_bf16_skinny_splitk_noalloc. */
#define SGEMM_NOALLOC_SCRATCH_BYTES (4u << 20)

/* Split-K GEMM that allocates nothing.  The paper has no counterpart: this
 * entry point exists for callers that cannot allocate device memory when they
 * run the GEMM (code under a memory manager that owns all device memory,
 * plugins or embedded runtimes that may not grow their footprint after
 * start-up, latency-critical loops where a possibly synchronizing cudaMalloc
 * is not allowed).  It computes y = x . W^T exactly like sgemm_bf16_skinny_ex
 * with the plan sgemm_splitk_noalloc_plan(N, K, M, split_k, NULL, ...) returns
 * (bitwise-equal results), but keeps the FP32 partial sums in a fixed,
 * library-owned device array of SGEMM_NOALLOC_SCRATCH_BYTES (4 MiB) instead
 * of allocated scratch.
 * - The caller passes inputs and outputs as for sgemm_bf16_skinny_ex (device
 *   pointers, strides in elements); split_k must be >= 2.  The launch is
 *   plain (no launch flags).
 * - split_k * M * N * 4 bytes must fit SGEMM_NOALLOC_SCRATCH_BYTES; larger
 *   problems return SGEMM_ERR_UNSUPPORTED_SHAPE and launch nothing.
 * - The first call on a device does a one-time set-up with that device current
 *   (it looks up the array's device address).  That first call must come
 *   before any stream capture: made on a capturing stream it returns
 *   SGEMM_ERR_INVALID_ARG and enqueues nothing.  Later calls may be captured.
 * - The array lives in every GPU that loads the library until the process
 *   exits.  All calls on a device share it and it keeps what the last call
 *   left; nothing in it needs clearing, because each call writes every partial
 *   sum it later reads.  Calls that overlap on the GPU (other streams,
 *   concurrent graph launches) race on it: order them.
 * - Never calls cudaMalloc, cudaFree or any allocating routine. */
sgemm_status_t sgemm_bf16_skinny_splitk_noalloc(const sgemm_bf16_t *x, long long ldx,
                                                const sgemm_bf16_t *W, sgemm_bf16_t *y,
                                                long long ldy, int M, int N, int K, int split_k,
                                                sgemm_stream_t stream);

/* The plan sgemm_bf16_skinny_splitk_noalloc runs for (N, K, M, split_k): the
 * plan `selected` (NULL = sgemm_plan_select(N, K, M)) with split_k K splits
 * through scratch memory and a second-pass reduce.  Plans that do not split K
 * that way are replaced: a TMA + tcgen05 plan (SGEMM_VARIANT_TC05, whose split
 * reduces inside a cluster) by the CUDA-core streaming plan (variant
 * SGEMM_VARIANT_LDG_MIXFMA, 256 threads, 1 row per warp, 32 lanes per row,
 * k_unroll 8, 1 stage), and a cluster-split streaming plan
 * (SGEMM_VARIANT_LDG_CLUSTER) by the same configuration as variant
 * SGEMM_VARIANT_LDG_MIXFMA.  Pure host function.  Writes *out
 * and returns sgemm_plan_check of it for (M, N, K); SGEMM_ERR_INVALID_ARG for
 * a NULL out or split_k < 2. */
sgemm_status_t sgemm_splitk_noalloc_plan(int N, int K, int M, int split_k,
                                         const sgemm_plan_t *selected, sgemm_plan_t *out);

/* Reads and clears the device error word of the current device: bit 0 is set
 * when a kernel gave up a bounded wait for its data (SGEMM_VARIANT_TC05; the
 * outputs of that launch were written as NaN).
 * *flags = 0 when nothing went wrong.  The word is a static device variable
 * of the library (no allocation).  Synchronous (waits for the device); do not
 * call during stream capture. */
sgemm_status_t sgemm_device_errors(int *flags);

/* Static description of a status code (never NULL). */
const char *sgemm_status_string(sgemm_status_t status);

/* Library version, "major.minor.patch". */
const char *sgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SGEMM_SKINNY_H */
