// k_gemv.cu -- the row-parallel projection (GEMV) of every simulated rank,
// the producer of the AllReduce in a tensor-parallel decode layer.
//
// "vLLM distributed inference core" (page 2), section one: each layer's
// attention output projection and MLP down projection are split by rows
// over the ranks and end in an AllReduce of the partial results; section
// two: work that does not depend on the AllReduce's result can run while it
// is in flight -- the page's example is fetching the next layer's memory.
// Here the next projection's weights are that work: the kernel is launched
// as a programmatic dependent of the AllReduce before it, prefetches the
// first rows of its weight tile into L2 (weights never depend on the
// AllReduce), and only then waits for the AllReduce to complete before it
// reads its input.  It does not let the kernel after it launch early: an
// AllReduce whose CTAs become resident while the projection still streams
// slowed a decode step by 4% on GB300, so the next AllReduce starts when the
// projection completes.
//
// What it computes, rank r, column j: y[j] = bf16( P_0 + P_1 + ... + P_7 ),
// P_s = (((+0 + p_i0) + p_i0+1) + ...) over the rows i of segment s (rows
// [s*c, min(k, (s+1)*c)), c = ceil(k / 8)) in row order, p_i = x[i] * W[i][j]
// rounded to binary32 (exact unless it under- or overflows); every add is a
// binary32 add rounded to nearest even; one rounding to bf16.
//
// Layout: CTA (r, t) covers columns [256 t, 256 t + 256) of rank r; warp s
// streams segment s, lane l holds columns 256 t + 8 l .. + 7 (one 16-byte
// load of a weight row), 8 rows in flight per lane.  The 8 segment sums meet
// in shared memory and thread j folds them for its column.  HBM-bound: k*h*2
// weight bytes per rank per call.
#include "sfar_gemv.h"
#include "sfar_prims.cuh"

namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Read-only loads as compiler builtins (not volatile asm), so that the eight
// rows of a step are all in flight before the first one is used.
__device__ __forceinline__ float ld_bf16(const uint16_t *p)
{
    return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p)) << 16);
}
__device__ __forceinline__ uint4 ld_w16(const uint16_t *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }

// acc[c] += x * W[c] for the 8 columns of one 16-byte weight vector
__device__ __forceinline__ void madd8(float *acc, float x, const uint4 &wv)
{
    acc[0] = __fadd_rn(acc[0], __fmul_rn(x, bf16_lo(wv.x)));
    acc[1] = __fadd_rn(acc[1], __fmul_rn(x, bf16_hi(wv.x)));
    acc[2] = __fadd_rn(acc[2], __fmul_rn(x, bf16_lo(wv.y)));
    acc[3] = __fadd_rn(acc[3], __fmul_rn(x, bf16_hi(wv.y)));
    acc[4] = __fadd_rn(acc[4], __fmul_rn(x, bf16_lo(wv.z)));
    acc[5] = __fadd_rn(acc[5], __fmul_rn(x, bf16_hi(wv.z)));
    acc[6] = __fadd_rn(acc[6], __fmul_rn(x, bf16_lo(wv.w)));
    acc[7] = __fadd_rn(acc[7], __fmul_rn(x, bf16_hi(wv.w)));
}

}  // namespace

__global__ void __launch_bounds__(SFAR_GEMV_SEGMENTS * 32, 2) k_gemv(const __grid_constant__ SfarGemvArgs g)
{
    __shared__ float part[SFAR_GEMV_SEGMENTS][SFAR_GEMV_COLS];
    const int r = blockIdx.x / g.tiles, t = blockIdx.x - r * g.tiles;
    const int lane = threadIdx.x & 31, s = threadIdx.x >> 5;
    const unsigned long long h = g.h;
    const unsigned long long c0 = (unsigned long long)t * SFAR_GEMV_COLS + lane * 8ull;
    const bool col_ok = c0 < h;
    const unsigned long long i0 = (unsigned long long)s * g.seg;
    const unsigned long long i1 = i0 + g.seg < g.k ? i0 + g.seg : g.k;
    const uint16_t *W = static_cast<const uint16_t *>(g.w[r]);
    const uint16_t *x = static_cast<const uint16_t *>(g.x[r]);

    // the first rows of this warp's weight slice, one prefetch per 128-byte line
    if (col_ok && (lane & 7) == 0) {
        const unsigned long long pe = i0 + g.prefetch < i1 ? i0 + g.prefetch : i1;
        for (unsigned long long i = i0; i < pe; ++i)
            prefetch_l2(W + i * h + c0);
    }
    pdl_wait();

    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (col_ok) {
        unsigned long long i = i0;
        for (; i + 8 <= i1; i += 8) {
            uint4 wv[8];
            float xv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                wv[u] = ld_w16(W + (i + u) * h + c0);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                xv[u] = ld_bf16(x + i + u);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                madd8(acc, xv[u], wv[u]);
        }
        for (; i < i1; ++i)
            madd8(acc, ld_bf16(x + i), ld_w16(W + i * h + c0));
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        part[s][lane * 8 + c] = acc[c];
    __syncthreads();
    const unsigned long long col = (unsigned long long)t * SFAR_GEMV_COLS + threadIdx.x;
    if (col < h) {
        float y = part[0][threadIdx.x];
#pragma unroll
        for (int q = 1; q < SFAR_GEMV_SEGMENTS; ++q)
            y = __fadd_rn(y, part[q][threadIdx.x]);
        const unsigned short b = __bfloat16_as_ushort(__float2bfloat16_rn(y));
        asm volatile("st.global.u16 [%0], %1;" ::"l"(static_cast<uint16_t *>(g.y[r]) + col), "h"(b) : "memory");
    }
}

const void *sfar_kernel_gemv() { return (const void *)k_gemv; }
