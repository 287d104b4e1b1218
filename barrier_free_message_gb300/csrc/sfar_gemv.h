// sfar_gemv.h -- parameters of the row-parallel projection kernel that
// produces the AllReduce's inputs in a tensor-parallel decode layer.
#pragma once
#include "sfar_internal.h"

#define SFAR_GEMV_SEGMENTS 8          // K-segments, one per warp of a CTA
#define SFAR_GEMV_COLS 256            // columns per CTA: 32 lanes x 8 bf16

struct SfarGemvArgs {
    const void *x[SFAR_MAX_R];        // [k] bf16 per rank
    const void *w[SFAR_MAX_R];        // [k][h] bf16 per rank, row-major
    void *y[SFAR_MAX_R];              // [h] bf16 per rank
    unsigned long long k, h;
    unsigned long long seg;           // rows per segment: ceil(k / 8)
    unsigned long long prefetch;      // rows of each segment prefetched into L2 before the launch wait
    int tiles;                        // column tiles per rank: ceil(h / 256)
};

const void *sfar_kernel_gemv();
