// k_fused.cu -- the fused AllReduce + residual add + RMS normalisation with
// 16-byte units, and the lookup of every variant.
#include "fused_kernel.cuh"

SFAR_FUSED_TABLE(sfar_kernel_fused_u16, 16)

const void *sfar_kernel_fused(int dt, int wide, int allreduce, int test, int batch, int unit)
{
    return unit == 8 ? sfar_kernel_fused_u8(dt, wide, allreduce, test, batch)
                     : sfar_kernel_fused_u16(dt, wide, allreduce, test, batch);
}
