// k_fused8.cu -- the fused AllReduce + residual add + RMS normalisation with
// 8-byte units (AllReduce of rows of up to 16 KB, one row per cluster), in its
// own translation unit so that the two unit sizes compile in parallel.
#include "fused_kernel.cuh"

SFAR_FUSED_TABLE(sfar_kernel_fused_u8, 8)
