// sfar_gemv.h -- parameters of the row-parallel projection kernel that
// produces the AllReduce's inputs in a tensor-parallel decode layer.
#pragma once
#include <cuda.h>

#include "sfar_internal.h"

#define SFAR_GEMV_COLS 256            // columns per CTA (512 bytes of a weight row)
#define SFAR_GEMV_CPT 2               // columns per thread: 2 or 4
#define SFAR_GEMV_THREADS (SFAR_GEMV_COLS / SFAR_GEMV_CPT)
#define SFAR_GEMV_ROWS 64             // weight rows per stage of the shared-memory ring (one TMA box)
#define SFAR_GEMV_STAGES 3            // stages in the ring; STAGES - 1 are in flight
#define SFAR_GEMV_SMEM (SFAR_GEMV_STAGES * SFAR_GEMV_ROWS * SFAR_GEMV_COLS * 2)

struct SfarGemvArgs {
    // W of every rank as a 2-D tensor map: h bf16 columns (innermost, stride 1)
    // by k rows (stride 2 h bytes), box SFAR_GEMV_COLS x SFAR_GEMV_ROWS, no
    // swizzle, zeros outside the matrix
    alignas(64) CUtensorMap wmap[SFAR_MAX_R];
    const void *x[SFAR_MAX_R];        // [k] bf16 per rank
    void *y[SFAR_MAX_R];              // [h] bf16 per rank
    SfarCtl *ctl;                     // the handle's status block: a copy wait that gives up is recorded here
    unsigned long long k, h;
    int pre;                          // stages whose copies are issued before the launch wait (0 .. STAGES - 1)
    int tiles;                        // column tiles per rank: ceil(h / SFAR_GEMV_COLS)
};

const void *sfar_kernel_gemv();
