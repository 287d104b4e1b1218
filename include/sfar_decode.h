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
 * the AllReduce is in flight, prefetches the first rows of its weights into
 * L2 (weights never depend on the AllReduce), and only then waits for the
 * AllReduce to complete before it reads its input.  It does not let the
 * kernel after it start early (an AllReduce resident during the projection's
 * weight stream slowed the decode step), so whatever follows sees plain
 * stream order.
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
 * bf16; hidden must be a multiple of 8.  Per output j the sum is fixed (it is
 * not given by the pages): each product x[i] * w[i][j] rounded to binary32
 * (exact unless it under- or overflows), the k rows cut into 8 segments of
 * ceil(k / 8) consecutive rows, each segment summed in row order into a
 * binary32 accumulator that starts at +0, the 8 segment sums folded in
 * segment order, one rounding to bf16 (nearest even).
 * prefetch_rows: rows of each segment whose weights are prefetched into L2
 * before the kernel waits for its predecessor (0 = none; capped at the
 * segment length).  Enqueues one kernel on stream s; capturable.  Returns
 * SFAR_ERR_INVALID for a bad argument (nothing enqueued), SFAR_ERR_CUDA if
 * the launch fails.
 */
sfar_status sfar_rowpar_gemv(sfar_t *h, const void *const x[], const void *const w[], void *const y[], size_t k,
                             size_t hidden, size_t prefetch_rows, sfar_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* SFAR_DECODE_H */
