/*
 * sfar_decode.h -- the producer of the AllReduce in a tensor-parallel decode
 * layer: the row-parallel projection (GEMV) of every simulated rank.
 *
 * "vLLM distributed inference core" (page 2), section one: with tensor
 * parallelism, each transformer layer's attention output projection and MLP
 * down projection are split by rows over the ranks and end in an AllReduce
 * of the ranks' partial results (two per layer, 160 per token for 80
 * layers); section two: work that does not depend on the AllReduce's result
 * overlaps it, the page's example being the fetch of the next layer's memory;
 * section three: the projection runs on the compute stream and the
 * AllReduce after it.
 *
 * On one GPU with R simulated ranks the projection of every rank is one
 * kernel.  Launched after an AllReduce on the same stream (in the handle's
 * serial launch mode) it is a programmatic dependent of it: it starts while
 * the AllReduce is in flight, issues the copies of the first rows of its
 * weights into shared memory (weights never depend on the AllReduce), and
 * only then waits for the AllReduce to complete before it reads its input.
 * It does not let the kernel after it start early (an AllReduce resident
 * during the projection's weight stream slowed the decode step), so whatever
 * follows sees plain stream order.
 */
#ifndef SFAR_DECODE_H
#define SFAR_DECODE_H

#include "sfar.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * sfar_rowpar_gemv: for every rank r of the handle, y[r] = x[r] W[r]:
 *   x[r]: k bf16 (the rank's slice of the layer input), 2-byte aligned;
 *   w[r]: k x hidden bf16, row-major (row i = the weights of input i),
 *         16-byte aligned;
 *   y[r]: hidden bf16 (the partial sums the AllReduce adds), 16-byte
 *         aligned, overlapping no x or w.
 * HOST arrays of R DEVICE pointers, owned by the caller.  The handle must be
 * bf16; hidden must be a multiple of 8.  Per output j the sum is fixed (the
 * pages give none; this is the plain definition): each product
 * x[i] * w[i][j] rounded to binary32 (exact unless it under- or overflows),
 * added in row order (i = 0 first) to one binary32 accumulator that starts
 * at +0, each add rounded to nearest even, then one rounding to bf16
 * (nearest even).
 * prefetch_rows: rows of each CTA's weight tile whose copies into shared
 * memory are issued before the kernel waits for its predecessor, in whole
 * stages of 64 rows (0 = none; capped at 2 stages, 128 rows, the copies the
 * kernel issues before its first fold).  Returns SFAR_ERR_UNSUPPORTED if the
 * driver offers no tensor-map encoder (the weights are read by 2-D TMA
 * copies); k and hidden must be below 2^31.  Enqueues one kernel on stream s;
 * capturable.  Returns SFAR_ERR_INVALID for a bad argument (nothing
 * enqueued), SFAR_ERR_CUDA if the launch fails.  On the device every wait
 * for a weight copy is bounded by the handle's timeout; one that gives up
 * is recorded in the handle's status (sfar_status_get: SFAR_ERR_TIMEOUT,
 * where = SFAR_WAIT_COPY, rank and CTA of the projection) and that CTA's
 * 256 columns of y are left unwritten.
 */
sfar_status sfar_rowpar_gemv(sfar_t *h, const void *const x[], const void *const w[], void *const y[], size_t k,
                             size_t hidden, size_t prefetch_rows, sfar_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* SFAR_DECODE_H */
