// k_gemv.cu -- the row-parallel projection (GEMV) of every simulated rank,
// the producer of the AllReduce in a tensor-parallel decode layer.
//
// "vLLM distributed inference core" (page 2), section one: each layer's
// attention output projection and MLP down projection are split by rows
// over the ranks and end in an AllReduce of the partial results; section
// two: work that does not depend on the AllReduce's result can run while it
// is in flight -- the page's example is fetching the next layer's memory.
// Here the next projection's weights are that work: the kernel is launched
// as a programmatic dependent of the AllReduce before it, issues the copies
// of the first rows of its weight tile into shared memory (weights never
// depend on the AllReduce), and only then waits for the AllReduce to
// complete before it reads its input.  It does not let the kernel after it
// launch early: an AllReduce whose CTAs become resident while the projection
// still streams slowed a decode step by 4% on GB300, so the next AllReduce
// starts when the projection completes.
//
// What it computes, rank r, column j: y[j] = bf16( (((+0 + p_0) + p_1) + ...)
// + p_(k-1) ), p_i = x[i] * W[i][j] rounded to binary32 (exact unless it
// under- or overflows); every add a binary32 add rounded to nearest even; one
// rounding to bf16.  The sum of a column is one chain of k dependent adds,
// so the parallelism is across columns: R * h chains.
//
// Layout: CTA (r, t) covers columns [256 t, 256 t + 256) of rank r and all k
// rows; thread l folds columns 256 t + 2 l and 256 t + 2 l + 1.  The weight
// tile streams through a ring of 3 shared-memory stages of 64 rows (32 KB),
// each filled by one 2-D TMA tensor copy (a box of 64 rows x 256 columns,
// zeros past the matrix's last row or column) that thread 0 issues and whose
// completion is counted in bytes on the slot's mbarrier: two stages (64 KB
// per CTA, two CTAs per SM) are in flight while the threads fold the third,
// and the folding threads spend no instructions on copies.  (Copies of one
// 512-byte row each, or 16 bytes per thread, cost more than the fold: the
// first capped the stream near 3.8 TB/s, the second took 40% of the issue
// slots.)  Every thread loads its stage's weight words and the stage's x
// (binary32, staged in shared memory by warp 0 one group of 256 rows ahead)
// before its first add, so the adds wait only on one another.  One CTA-wide
// barrier per stage frees the slot of the stage before.  Every wait for a
// copy is bounded; one that gives up is recorded in the handle's status
// block, and the CTA waits (bounded again) for the copies it still has in
// flight before it returns.  HBM-bound: k*h*2 weight bytes per rank per call.
#include "sfar_gemv.h"
#include "sfar_prims.cuh"

namespace {

constexpr int kCols = SFAR_GEMV_COLS, kThreads = SFAR_GEMV_THREADS, kCpt = SFAR_GEMV_CPT;
constexpr int kRows = SFAR_GEMV_ROWS, kStages = SFAR_GEMV_STAGES;
constexpr int kRowBytes = kCols * 2;                    // one row of a tile in the ring
constexpr int kStageBytes = kRows * kRowBytes;
constexpr int kGroupRows = 32 * 8;                      // rows of x one load of warp 0 covers: 8 per lane
constexpr int kGroupStages = kGroupRows / kRows;
static_assert(kGroupRows % kRows == 0 && kRows % 4 == 0 && kStages >= 2, "stages tile the x groups");
static_assert((kCpt == 2 || kCpt == 4) && kThreads * kCpt == kCols && kThreads % 32 == 0, "2 or 4 columns per thread");

// a thread's kCpt bf16 weights of one row
template <int C> struct WVec;
template <> struct WVec<2> {
    using T = uint32_t;
    static __device__ __forceinline__ float at(const T &v, int c) { return __uint_as_float(c ? v & 0xffff0000u : v << 16); }
};
template <> struct WVec<4> {
    using T = uint2;
    static __device__ __forceinline__ float at(const T &v, int c)
    {
        const uint32_t w = c < 2 ? v.x : v.y;
        return __uint_as_float(c & 1 ? w & 0xffff0000u : w << 16);
    }
};
using W = WVec<kCpt>;

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for phase `parity` of a slot's mbarrier, at most limit_ns; false if it gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 127u) == 0 && globaltimer() - t0 > limit_ns)
            return false;
    }
}
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// box (x, y) = (first column, first row) of a 2-D tensor map into shared memory
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar,
                                            uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

// The tile of one CTA: columns [c0, c0 + 256) of every row of W.
struct Tile {
    const CUtensorMap *map;        // W of the CTA's rank
    int c0;
    uint32_t ring;                 // shared-memory address of slot 0
    uint32_t full;                 // shared-memory address of slot 0's mbarrier (8 bytes per slot)
    uint64_t pol;
};

// By one thread: the copy of stage q (rows [R q, R q + R), R rows per stage;
// rows past k and columns past h arrive as zeros) into slot s.  The box is
// always whole, so the slot expects all of its bytes.
__device__ __forceinline__ void issue_stage(const Tile &t, unsigned long long q, int s)
{
    const uint32_t bar = t.full + 8u * s;
    mbar_expect_tx(bar, kStageBytes);
    tma_load_2d(t.ring + (uint32_t)(s * kStageBytes), t.map, t.c0, (int)(q * kRows), bar, t.pol);
}

// x of rows [256 G, 256 G + 256): lane l takes rows 256 G + 8 l .. + 7 (0 past k)
__device__ __forceinline__ void load_x(float (&xv)[8], const uint16_t *x, unsigned long long k, unsigned long long G,
                                       int lane)
{
    const unsigned long long i0 = G * kGroupRows + 8ull * lane;
#pragma unroll
    for (int e = 0; e < 8; ++e)
        xv[e] = i0 + e < k ? __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(x + i0 + e)) << 16)
                           : 0.f;
}
__device__ __forceinline__ void store_x(float *xs, const float (&xv)[8], int lane)
{
    reinterpret_cast<float4 *>(xs)[2 * lane] = make_float4(xv[0], xv[1], xv[2], xv[3]);
    reinterpret_cast<float4 *>(xs)[2 * lane + 1] = make_float4(xv[4], xv[5], xv[6], xv[7]);
}

// Folds the first n rows of a stage into a[], in row order.  w: this thread's
// weights in the stage's row 0; xr: the x of the stage's rows (shared memory,
// binary32).  All loads are issued before the first add.
template <bool FULL>
__device__ __forceinline__ void fold_stage(float (&a)[kCpt], const unsigned char *w, const float *xr, int n)
{
    typename W::T wv[kRows];
    float xv[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u)
        wv[u] = *reinterpret_cast<const typename W::T *>(w + u * kRowBytes);
#pragma unroll
    for (int u = 0; u < kRows; u += 4) {
        const float4 q = *reinterpret_cast<const float4 *>(xr + u);
        xv[u] = q.x;
        xv[u + 1] = q.y;
        xv[u + 2] = q.z;
        xv[u + 3] = q.w;
    }
#pragma unroll
    for (int u = 0; u < kRows; ++u)
        if (FULL || u < n) {
#pragma unroll
            for (int c = 0; c < kCpt; ++c)
                a[c] = __fadd_rn(a[c], __fmul_rn(xv[u], W::at(wv[u], c)));
        }
}

}  // namespace

__global__ void __launch_bounds__(SFAR_GEMV_THREADS, 2) k_gemv(const __grid_constant__ SfarGemvArgs g)
{
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(16) float xs[2][kGroupRows];      // x of two groups of rows, as binary32
    __shared__ __align__(8) unsigned long long full[kStages];
    const int r = blockIdx.x / g.tiles, tt = blockIdx.x - r * g.tiles;
    const int tid = threadIdx.x, lane = tid & 31;
    const unsigned long long c0 = (unsigned long long)tt * kCols;
    const unsigned long long nst = (g.k + kRows - 1) / kRows;
    Tile t;
    t.map = &g.wmap[r];
    t.c0 = (int)c0;
    t.ring = smem_u32(ring);
    t.full = smem_u32(full);
    t.pol = policy_evict_first();

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s)
            mbar_init(t.full + 8u * s, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    __syncthreads();
    // the first stages (slots 0 .. STAGES - 2); g.pre of them before the wait
    // for the kernel before (weights never depend on it)
    for (int q = 0; q < kStages - 1; ++q) {
        if (q == g.pre)
            pdl_wait();
        if (tid == 0 && (unsigned long long)q < nst)
            issue_stage(t, q, q);
    }
    if (g.pre >= kStages - 1)
        pdl_wait();
    const unsigned long long limit_ns = ld_relaxed_u64(&g.ctl->timeout_ns);

    // warp 0 keeps x one group ahead: groups 0 and 1 in shared memory, group 2 in registers
    const uint16_t *x = static_cast<const uint16_t *>(g.x[r]);
    float xn[8];
    if (tid < 32) {
        float x0[8];
        load_x(x0, x, g.k, 0, lane);
        load_x(xn, x, g.k, 1, lane);
        store_x(xs[0], x0, lane);
        store_x(xs[1], xn, lane);
        load_x(xn, x, g.k, 2, lane);
    }
    const bool live = c0 + 32ull * kCpt * (tid >> 5) < g.h;       // the warp has a column below h
    const unsigned char *mine = ring + tid * (kCpt * 2);
    float a[kCpt];
#pragma unroll
    for (int c = 0; c < kCpt; ++c)
        a[c] = 0.f;
    int rd = 0;                                             // slot of stage q
    uint32_t ph = 0;                                        // its phase parity
    unsigned long long q = 0;
    for (; q < nst; ++q) {
        const int gave_up = mbar_wait_bounded(t.full + 8u * rd, ph, limit_ns) ? 0 : 1;
        // stage q is in place; every thread is done with stage q - 1, so its
        // slot is free, and at a group's first stage so is the x buffer of the
        // group before
        if (__syncthreads_or(gave_up))
            break;
        const unsigned long long G = q / kGroupStages;
        const int j = (int)(q - G * kGroupStages);
        if (tid == 0 && q + kStages - 1 < nst)
            issue_stage(t, q + kStages - 1, rd == 0 ? kStages - 1 : rd - 1);
        if (tid < 32 && j == 0 && G > 0) {
            store_x(xs[(G + 1) & 1], xn, lane);             // read from the next group's first stage on
            load_x(xn, x, g.k, G + 2, lane);
        }
        if (live) {
            const unsigned char *w = mine + rd * kStageBytes;
            const float *xr = xs[G & 1] + j * kRows;
            const unsigned long long left = g.k - q * kRows;
            if (left >= (unsigned long long)kRows)
                fold_stage<true>(a, w, xr, kRows);
            else
                fold_stage<false>(a, w, xr, (int)left);
        }
        if (++rd == kStages) {
            rd = 0;
            ph ^= 1u;
        }
    }
    if (q < nst) {
        // a copy wait gave up: record it, and let the copies still in flight
        // (stages q .. q + STAGES - 2) land before the shared memory is released
        if (tid == 0) {
            sfar_record_fault(g.ctl, r, tt, -1, 0, SFAR_WAIT_COPY);
            for (unsigned long long p = q; p < nst && p < q + kStages - 1; ++p)
                mbar_wait_bounded(t.full + 8u * (uint32_t)(p % kStages), (uint32_t)((p / kStages) & 1ull), limit_ns);
        }
        return;
    }
    const unsigned long long col = c0 + (unsigned long long)kCpt * tid;
    if (col < g.h) {
        uint32_t v[kCpt / 2];
#pragma unroll
        for (int c = 0; c < kCpt / 2; ++c)
            v[c] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a[2 * c])) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(a[2 * c + 1])) << 16);
        uint16_t *dst = static_cast<uint16_t *>(g.y[r]) + col;
        if (kCpt == 2)
            asm volatile("st.global.u32 [%0], %1;" ::"l"(dst), "r"(v[0]) : "memory");
        else
            asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(dst), "r"(v[0]), "r"(v[kCpt / 2 - 1]) : "memory");
    }
}

const void *sfar_kernel_gemv() { return (const void *)k_gemv; }
