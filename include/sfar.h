/*
 * sfar.h -- libsfar: barrier-free small-message AllReduce for R simulated
 * ranks on one GB300 (sm_103a).
 *
 * The operation (all calls below): every rank r holds a vector in[r] of n
 * elements; afterwards every out[r] holds the element-wise sum over the R
 * ranks.  "Every Microsecond Counts" (page 1), section "Tensor parallelism
 * and AllReduce", defines the collective (partial results of all GPUs summed
 * and handed back to all); section "Unified primitives and API design"
 * defines recvReduce (receive every peer's value and reduce it in registers).
 * The sum is a left fold in rank order 0..R-1 with binary32 accumulation
 * (round to nearest even after every add) and one rounding to the output
 * type, so the result is unique bit for bit and identical on every rank,
 * whatever the protocol -- except SFAR_LL128_ATOMIC, whose binary32
 * accumulation happens in the order of the hardware atomics (see there).
 *
 * Simulated ranks: rank r is a group of CTAs of one kernel with its own
 * receive buffers in HBM; ranks exchange data only by stores into each
 * other's buffers and synchronise only through flags in global memory.
 *
 * Threading: a handle may be used from one host thread at a time.  All
 * device work is asynchronous on the caller's stream and can be captured in
 * a CUDA graph (no allocation, no synchronisation inside sfar_allreduce).
 */
#ifndef SFAR_H
#define SFAR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *sfar_stream_t;

typedef struct sfar sfar_t;

typedef enum {
    SFAR_BF16 = 0, /* 2-byte elements, bfloat16 */
    SFAR_FP32 = 1  /* 4-byte elements, IEEE binary32 */
} sfar_dtype;

/*
 * Protocols.  Sources: "Every Microsecond Counts" (page 1), sections
 * "Global memory barriers" (the two barriers), "Four barrier-free mechanisms"
 * (LL, sentinel, double buffering, LL128) and "Unified primitives and API
 * design" (one-shot and two-shot variants, table of variants); "SiFAR"
 * (page 3), sections "Limits of existing algorithms" (one-shot with top and
 * bottom barrier, two-shot) and "Technique 1" (double buffering removes the
 * bottom barrier).
 */
typedef enum {
    SFAR_BASELINE = 0,    /* one-shot, one receive buffer, top AND bottom barrier      */
    SFAR_DB = 1,          /* one-shot, double-buffered by epoch parity, ready flags
                             (top barrier) only: the bottom barrier is gone           */
    SFAR_LL = 2,          /* one-shot, LL packets: 8-byte words {4 B data, 4 B flag}  */
    SFAR_LL128 = 3,       /* one-shot, 128-byte lines: 4 B flag + 124 B payload       */
    SFAR_SENTINEL = 4,    /* one-shot, receive buffers prefilled with a NaN pattern   */
    SFAR_TWOSHOT = 5,     /* reduce-scatter + all-gather over LL128 lines, double
                             buffered (medium messages)                               */
    SFAR_TWOSHOT_TMA = 6, /* reduce-scatter + all-gather straight from the inputs to
                             the outputs with TMA bulk copies (large messages)        */
    SFAR_LL128_ATOMIC = 7, /* reduce-scatter by hardware atomic adds into 128-byte
                             lines whose first word counts the arrivals, then an
                             all-gather over flagged lines (page 1, "Four
                             barrier-free mechanisms", part 4).  NOT bit-exact: the
                             binary32 accumulation runs in the atomics' order, and
                             each element lies within 2 (R-1) 2^-24 sum|x| +
                             2 R 2^-126 of the exact sum before its one rounding to
                             the output type (exact when every partial sum is
                             representable, e.g. small integers).  Identical on
                             every rank.                                               */
    SFAR_TWOSHOT_SENTINEL = 8 /* reduce-scatter + all-gather over sentinel-prefilled,
                                 double-buffered receive buffers: the pages' two-phase
                                 LLBuffer algorithm for 64 KB - 1 MB (page 1, "Unified
                                 primitives and API design", table of variants).  Inputs
                                 must not contain the sentinel pattern (as SFAR_SENTINEL) */
} sfar_proto;

#define SFAR_NUM_PROTOS 9

typedef int sfar_status;
#define SFAR_OK 0
#define SFAR_ERR_INVALID 1     /* bad argument (rank count, size, pointer, alignment, overlap) */
#define SFAR_ERR_CUDA 2        /* a CUDA runtime call failed (launch, copy, query)            */
#define SFAR_ERR_OOM 3         /* device or pinned allocation failed in sfar_create           */
#define SFAR_ERR_TIMEOUT 4     /* a bounded wait on the device gave up (see sfar_fault)       */
#define SFAR_ERR_UNSUPPORTED 5 /* this device cannot run the kernels (not sm_103, or the grid
                                  cannot be co-resident)                                       */
#define SFAR_ERR_POISONED 6    /* an earlier device-side failure; call sfar_reset             */

/* Where a bounded device wait gave up (sfar_fault.where). */
#define SFAR_WAIT_DONE 1      /* overlap mode: previous call of the same rank/CTA      */
#define SFAR_WAIT_LL 2        /* LL packet flag                                        */
#define SFAR_WAIT_SENTINEL 3  /* sentinel-prefilled slot still holds the sentinel      */
#define SFAR_WAIT_READY 4     /* ready flag / top barrier                              */
#define SFAR_WAIT_BOTTOM 5    /* bottom barrier                                        */
#define SFAR_WAIT_LL128 6     /* LL128 line flag (one-shot)                            */
#define SFAR_WAIT_RS 7        /* two-shot reduce-scatter line flag                     */
#define SFAR_WAIT_AG 8        /* two-shot all-gather line flag                         */
#define SFAR_WAIT_ARRIVE 9    /* TMA / two-shot fused: peer arrival (top barrier)      */
#define SFAR_WAIT_COMPLETE 10 /* TMA / two-shot fused: owner completion flags          */
#define SFAR_WAIT_COPY 11     /* TMA path or projection: bulk copy completion          */
#define SFAR_WAIT_COUNTER 12  /* atomic path: a line's arrival counter stayed below R  */
#define SFAR_WAIT_CLUSTER 13  /* fused normalisation: a cluster peer's row statistics
                                 (8 times the limit: every peer always sends); with
                                 SFAR_ERR_UNSUPPORTED, the grid had no clusters       */

typedef struct {
    sfar_status code; /* SFAR_OK or SFAR_ERR_TIMEOUT                          */
    int rank;         /* simulated rank whose wait gave up                    */
    int cta;          /* CTA index within that rank                           */
    int peer;         /* rank it was waiting for (-1 if not one rank)         */
    uint32_t epoch;   /* call epoch (1 for the handle's first call, +1 per call) */
    int where;        /* SFAR_WAIT_*                                          */
} sfar_fault;

/*
 * sfar_create: a handle for R simulated ranks (2 <= R <= 16) on the current
 * CUDA device, for messages of up to max_bytes per rank (> 0) of type dt.
 * Allocates, on the current device, the receive regions of every protocol
 * (double-buffered: [rank][parity][sender][wire bytes]; the sentinel region
 * prefilled with all-ones), the flag arrays, one call counter per rank (the
 * epoch of every call) and a status block, and zero-initialises them.  The
 * receive-buffer
 * protocols (every protocol but SFAR_TWOSHOT_TMA) handle up to
 * min(max_bytes, 2 MiB) per rank; SFAR_TWOSHOT_TMA handles up to max_bytes.
 * The library owns everything it allocates.  Returns NULL on error and sets
 * the calling thread's sfar_last_error(): SFAR_ERR_INVALID (bad R, max_bytes
 * or dt: checked before any CUDA call), SFAR_ERR_UNSUPPORTED (device is not
 * sm_103), SFAR_ERR_OOM, SFAR_ERR_CUDA.
 */
sfar_t *sfar_create(int R, size_t max_bytes, sfar_dtype dt);

/* The error of the calling thread's last failed sfar_create (thread-local). */
sfar_status sfar_last_error(void);

/*
 * sfar_allreduce: in and out are HOST arrays of R DEVICE pointers (owned by
 * the caller); in[r] and out[r] each hold n elements of the handle's dtype,
 * 16-byte aligned.  No output may overlap an input or another output.
 * n * element size must not exceed the protocol's limit (see sfar_create).
 * n == 0 is a no-op.  Enqueues ONE kernel on stream s and returns at once;
 * capturable in a CUDA graph.  Returns, without enqueuing anything,
 * SFAR_ERR_INVALID for a bad argument, SFAR_ERR_POISONED after a device-side
 * failure that sfar_status_get has reported, SFAR_ERR_UNSUPPORTED if the
 * grid the call needs cannot be co-resident (every CTA of a call waits on
 * others; the grid is sized for an idle device, and in the cooperative launch
 * mode of sfar_test.h the device places it whole or refuses it), and
 * SFAR_ERR_CUDA if the launch fails.  A device-side failure (a bounded wait giving up) does not show
 * here: it is recorded in the handle's status block (sticky) and every later
 * kernel of the handle exits at once; read it with sfar_status_get.
 */
sfar_status sfar_allreduce(sfar_t *h, const void *const in[], void *const out[], size_t n,
                           sfar_proto p, sfar_stream_t s);

/*
 * sfar_status_get: reads the handle's device status block through a private
 * stream and returns its code (SFAR_OK; SFAR_ERR_TIMEOUT; or
 * SFAR_ERR_UNSUPPORTED with where = SFAR_WAIT_CLUSTER when a fused kernel
 * found itself launched without the thread-block clusters it was planned
 * for, e.g. by a tool replaying the launch, and ran nothing); fills *info if
 * info is not NULL.  It does not wait for the caller's streams: synchronise
 * them first to see the outcome of the work enqueued so far.  A non-OK code
 * poisons the handle on the host too, until sfar_reset.
 */
sfar_status sfar_status_get(sfar_t *h, sfar_fault *info);

/*
 * sfar_reset: enqueues on s the re-initialisation of every flag, epoch and
 * receive region (sentinel region re-seeded) and clears the status block and
 * the host-side poison.  The caller must ensure no kernel of this handle is
 * still running on another stream.
 */
sfar_status sfar_reset(sfar_t *h, sfar_stream_t s);

/* sfar_destroy: frees everything the handle owns; NULL is allowed.  The
 * caller must have synchronised all work enqueued with the handle. */
void sfar_destroy(sfar_t *h);

/* A static, human-readable string for a status code. */
const char *sfar_strerror(sfar_status st);

/* Launch geometry of a call (for reports): CTAs per rank and threads per
 * CTA the kernel would use for n elements under protocol p. */
sfar_status sfar_query_launch(const sfar_t *h, size_t n, sfar_proto p, int *ctas_per_rank,
                              int *threads_per_cta);

/* Largest n * element size per rank that protocol p accepts on this handle. */
size_t sfar_max_bytes(const sfar_t *h, sfar_proto p);

/*
 * sfar_allreduce_add_rmsnorm: the AllReduce of sfar_allreduce(..., SFAR_LL,
 * ...) followed, in the same kernel, by the residual add and the RMS
 * normalisation that come next in a decode layer ("vLLM distributed
 * inference core" (page 2), sections one and two: the normalisation runs on
 * the compute stream right after the AllReduce of the attention output and
 * of the MLP down projection).  The pages give no formula; the one
 * implemented, with every rounding fixed so the result is unique bit for bit
 * whatever the launch geometry, is, per rank r and row i of `hidden`
 * elements (T = the handle's dtype):
 *   a   = the AllReduce result of the row, in T (as sfar_allreduce stores it);
 *   z   = T(a + residual[r])                      binary32 add;
 *   ms  = ldexp(float(S) / hidden, 2E - F), S = the sum of z^2 over the row
 *         in units of 2^(2E - F), each term truncated to a whole unit (2^E
 *         the smallest power of two above every |z|, F = 53 -
 *         ceil(log2 hidden)): an exact integer sum below 2^53, short of the
 *         exact sum of squares by less than 2^(2c - 51) of the largest square
 *         (c = ceil(log2 hidden)); float(S) and the division are binary32,
 *         each rounded once;
 *         a NaN in the row gives NaN, else an infinity gives +inf;
 *   y   = T((z * (1 / sqrt(ms + eps))) * weight)  each binary32 operation
 *         rounded to nearest even.
 * out[r] receives y and residual_out[r] receives z (rows x hidden each).
 * in, residual, out, residual_out: HOST arrays of R DEVICE pointers, each
 * buffer rows * hidden elements, row-major, 16-byte aligned; weight: one
 * device buffer of hidden elements shared by all ranks, 16-byte aligned.
 * hidden * element size must be a multiple of 16 and at most 128 KiB (64 KiB
 * for R > 8); rows * hidden * element size must not exceed
 * sfar_max_bytes(h, SFAR_LL).
 * residual_out[r] may be residual[r] (in place); otherwise no output may
 * overlap an input, the weight or another output.  rows == 0 is a no-op.
 * One kernel on stream s (thread-block clusters, one cluster per row at a
 * time); capturable; errors as for sfar_allreduce.  The kernel depends on
 * the shape, the result does not: the one-shot kernel over LL packets, or,
 * when that kernel would stack several rows on a cluster and rows are at
 * most 32 KB, a two-shot kernel ("SiFAR" (page 3), "Limits of existing
 * algorithms") in which the owner of a row reads it from every rank once and
 * writes every rank's z and y.
 */
sfar_status sfar_allreduce_add_rmsnorm(sfar_t *h, const void *const in[], const void *const residual[],
                                       const void *weight, void *const out[], void *const residual_out[],
                                       size_t rows, size_t hidden, float eps, sfar_stream_t s);

/*
 * sfar_add_rmsnorm: the same residual add and normalisation on its own:
 * a[r] is taken as rank r's AllReduce result (rows x hidden elements of the
 * handle's dtype).  The arguments, the definition and the rules are those of
 * sfar_allreduce_add_rmsnorm (minus the AllReduce and its size limit); it
 * uses none of the handle's buffers, only its rank count and dtype.  One
 * kernel on stream s.
 */
sfar_status sfar_add_rmsnorm(sfar_t *h, const void *const a[], const void *const residual[], const void *weight,
                             void *const out[], void *const residual_out[], size_t rows, size_t hidden, float eps,
                             sfar_stream_t s);

/*
 * sfar_allreduce_noalloc: the same AllReduce as sfar_allreduce(h, in, out, n,
 * SFAR_LL, s) on a handle of R ranks and type dt, for callers that cannot
 * allocate device memory at the moment they need it: code running under
 * stream capture (cudaMalloc is not allowed there), code inside a framework
 * whose allocator owns all device memory, and latency paths that cannot pay
 * for cudaMalloc's implicit synchronisation.  There is no counterpart in the
 * pages; it is a convenience of this library.
 *
 * No handle and no allocation: the kernel's working memory is one fixed
 * array of about 13 MiB compiled into the library, present on every GPU that
 * loads the library until the process exits.  in/out are host arrays of R
 * device pointers as for sfar_allreduce (16-byte aligned, no output
 * overlapping an input or another output).  Limits: 2 <= R <=
 * SFAR_NOALLOC_MAX_RANKS and n * element size <= SFAR_NOALLOC_MAX_BYTES;
 * anything larger returns SFAR_ERR_INVALID and enqueues nothing.
 *
 * The first call on each device sets the array up (finds its address,
 * checks that the grid fits, clears it) and synchronises stream s, so make
 * that first call before any stream capture; later calls only enqueue one
 * kernel and can be captured.  All calls share the array and it keeps what
 * the last call left (its call counters keep counting); calls whose kernels
 * overlap on the GPU, e.g. on two streams at once, race on it.  Returns
 * SFAR_ERR_UNSUPPORTED on a device that is not sm_103 and SFAR_ERR_CUDA if a
 * CUDA call fails.  A device-side failure (a bounded wait that gave up)
 * stays recorded in the array, and every later kernel then returns without
 * writing its outputs; sfar_noalloc_status reports it, after which calls
 * return SFAR_ERR_POISONED and enqueue nothing until the record is cleared.
 */
#define SFAR_NOALLOC_MAX_RANKS 8
#define SFAR_NOALLOC_MAX_BYTES 16384
sfar_status sfar_allreduce_noalloc(const void *const in[], void *const out[], int R, size_t n, sfar_dtype dt,
                                   sfar_stream_t s);

/*
 * sfar_noalloc_status: the outcome of the sfar_allreduce_noalloc calls made
 * so far on the current device, read from the fixed array's status block by
 * a synchronous copy (synchronise the streams of those calls first).  Returns
 * SFAR_OK, or SFAR_ERR_TIMEOUT if a bounded device wait of one of them gave
 * up, and fills *info (if not NULL) as sfar_status_get does.  With clear == 0
 * a reported failure poisons the entry point on this device: later
 * sfar_allreduce_noalloc calls return SFAR_ERR_POISONED.  With clear != 0 it
 * returns the recorded code, then erases the record and the poison, and
 * later calls compute again: the array's call counters stay consistent
 * across a failed call, so nothing else needs resetting.  Clear only while
 * no kernel of the entry point runs on the device.  SFAR_OK on a device that
 * has made no such call; SFAR_ERR_CUDA if a copy fails.  Like the entry point
 * itself, it has no counterpart in the pages.
 */
sfar_status sfar_noalloc_status(sfar_fault *info, int clear);

#ifdef __cplusplus
}
#endif

#endif /* SFAR_H */
