// sfar_fused.h -- parameters of the fused AllReduce + residual add + RMS
// normalisation kernels: a second kernel parameter next to SfarArgs.
#pragma once
#include "sfar_internal.h"

#define SFAR_NORM_VMAX 4          // 16-byte vectors of one row per thread
#define SFAR_NORM_CLMAX 8         // CTAs per cluster (portable cluster size)
#define SFAR_NORM_THREADS 256     // upper bound of threads per CTA

struct SfarNormArgs {
    const void *res[SFAR_MAX_R];  // residual stream of each rank (rows x hidden)
    void *res_out[SFAR_MAX_R];    // z = T(a + res) of each rank (may be res itself)
    const void *weight;           // hidden elements, shared by all ranks
    unsigned long long rows, hidden;
    float eps;
    int G;                        // clusters per rank (rows g, g + G, ...)
    int CL;                       // CTAs per cluster: a row is spread over one cluster
    int F;                        // fixed-point fraction bits of the sum of squares
    int vpt;                      // vectors of a row per thread: ceil(hidden vectors / (CL * threads))
    int B;                        // rows per statistics round: 1, or up to 4 when vpt == 1
};

// dt: 0 bf16, 1 fp32; wide: R > 8; allreduce: 1 = AllReduce over LL packets
// first, 0 = the normalisation of a given AllReduce result; test: knobs;
// batch: rows per statistics round (1, or up to 4 when every thread holds one
// unit of each row); unit: bytes per unit, 16 or 8.
const void *sfar_kernel_fused(int dt, int wide, int allreduce, int test, int batch, int unit);
const void *sfar_kernel_fused_u16(int dt, int wide, int allreduce, int test, int batch);
const void *sfar_kernel_fused_u8(int dt, int wide, int allreduce, int test, int batch);
// The two-shot fused kernel (rows of at most 32 KB, one 16-byte unit per
// thread): dt, wide and test as above.
const void *sfar_kernel_fused_ts(int dt, int wide, int test);
