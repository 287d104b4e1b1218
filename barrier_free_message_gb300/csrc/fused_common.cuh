// fused_common.cuh -- device helpers shared by the fused AllReduce + residual
// add + RMS normalisation kernels: the order-free row statistics (largest
// magnitude, exact integer sum of truncated squares), element lanes of a
// 16-byte vector, unit loads and stores, and the exchange of row statistics
// between the CTAs of a thread-block cluster (st.async into each other's
// shared memory, counted by mbarriers).
#pragma once
#include "sfar_fused.h"
#include "sfar_prims.cuh"

namespace {

__device__ __forceinline__ uint32_t mag_bits(float v) { return __float_as_uint(v) & 0x7fffffffu; }

// Largest magnitude of the first n bf16 elements of a 16-byte vector, as
// binary32 magnitude bits (a bf16's bits are the upper half of its binary32
// bits, and magnitude bits compare as unsigned integers): pairwise maxima of
// the 16-bit halves, then of the two halves left.  Lanes past n are cleared.
__device__ __forceinline__ uint32_t max_mag_bf16(const uint4 &z, int n)
{
    uint32_t w[4] = {z.x, z.y, z.z, z.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t keep = 2 * i + 1 < n ? 0x7fff7fffu : 2 * i < n ? 0x00007fffu : 0u;
        w[i] &= keep;
    }
    uint32_t a, b, m;
    asm("max.u16x2 %0, %1, %2;" : "=r"(a) : "r"(w[0]), "r"(w[1]));
    asm("max.u16x2 %0, %1, %2;" : "=r"(b) : "r"(w[2]), "r"(w[3]));
    asm("max.u16x2 %0, %1, %2;" : "=r"(m) : "r"(a), "r"(b));
    return max(m >> 16, m & 0xffffu) << 16;
}

// smallest E with |v| < 2^E for the finite nonzero magnitude bits m
__device__ __forceinline__ int exp_above(uint32_t m)
{
    const uint32_t eb = m >> 23;
    if (eb)
        return (int)eb - 126;
    return (31 - __clz((int)m)) - 148;
}

// floor(v^2 2^(F - 2E)) for finite v with |v| < 2^E: an integer below 2^F,
// from the binary32 fields (v = m 2^e2), exact
__device__ __forceinline__ unsigned long long sq_term(float v, int E, int F)
{
    const uint32_t b = mag_bits(v);
    if (b == 0)
        return 0ull;
    const uint32_t eb = b >> 23, fr = b & 0x7fffffu;
    const unsigned long long m = eb ? (fr | 0x800000u) : fr;
    const int e2 = eb ? (int)eb - 150 : -149;
    const int sh = 2 * e2 - 2 * E + F;
    const unsigned long long m2 = m * m;
    if (sh >= 0)
        return m2 << sh;
    return -sh >= 64 ? 0ull : (m2 >> (-sh));
}

// The same truncated square for values of at most 8 significant bits (bf16
// elements), in binary32: v is scaled by 2^k, k = floor(F/2) - E, in two
// exact steps (each factor within 2^-55 .. 2^87), so |v 2^k| < 2^26 and its
// square has at most 16 significant bits: exact whenever it is normal, and
// below 1 (truncating to 0 either way) when it is not.  The square, doubled
// when F is odd (exact), truncated to an integer is floor(v^2 2^(F - 2E)).
// The truncation reads the binary32 fields with integer operations: the
// float-to-64-bit-integer conversion ran slowly enough to cost the two-shot
// fused call (64 rows of 7168 bf16, R = 8) 20.9 instead of 17.0 us.
struct SqScale {
    float s1, s2;
    bool odd;
};
__device__ __forceinline__ SqScale sq_scale(int E, int F)
{
    const int k = (F >> 1) - E;
    const int k1 = k >> 1, k2 = k - k1;
    return {__int_as_float((127 + k1) << 23), __int_as_float((127 + k2) << 23), (F & 1) != 0};
}
__device__ __forceinline__ unsigned long long sq_term_narrow(float v, const SqScale &s)
{
    const float vs = __fmul_rn(__fmul_rn(v, s.s1), s.s2);
    float t = __fmul_rn(vs, vs);
    if (s.odd)
        t = __fmul_rn(t, 2.0f);
    // floor(t) for 0 <= t < 2^53 (t is never negative: it is a square).  With
    // t = m 2^(x - 150), m the 24-bit significand and x the exponent field,
    // x - 150 <= 29, so floor(t) = (m 2^32) >> (182 - x): one 64-bit shift.
    // For t < 1 (zero and subnormals included) the amount is at least 56 and
    // the result 0; amounts above 63 are clamped by shr.b64 to a result of 0.
    const uint32_t b = __float_as_uint(t);
    const unsigned long long m = (unsigned long long)((b & 0x7fffffu) | 0x800000u) << 32;
    unsigned long long r;
    asm("shr.b64 %0, %1, %2;" : "=l"(r) : "l"(m), "r"(182u - (b >> 23)));
    return r;
}

__device__ __forceinline__ float mean_square(uint32_t M, unsigned long long S, unsigned long long h, int F)
{
    if (M > 0x7f800000u)
        return __uint_as_float(0x7fffffffu);
    if (M == 0x7f800000u)
        return __uint_as_float(0x7f800000u);
    if (M == 0)
        return 0.f;
    const int E = exp_above(M);
    return ldexpf(__fdiv_rn(__ull2float_rn(S), (float)h), 2 * E - F);
}

// element lanes of a 16-byte vector as binary32
template <int DT> struct Vec;
template <> struct Vec<0> {
    static constexpr int N = 8;
    __device__ __forceinline__ static float get(const uint4 &x, int i)
    {
        const uint32_t w = i < 2 ? x.x : i < 4 ? x.y : i < 6 ? x.z : x.w;
        return __uint_as_float((i & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    __device__ __forceinline__ static uint4 pack(const float *f)
    {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * q]));
            const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(f[2 * q + 1]));
            w[q] = lo | (hi << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};
template <> struct Vec<1> {
    static constexpr int N = 4;
    __device__ __forceinline__ static float get(const uint4 &x, int i)
    {
        return __uint_as_float(i == 0 ? x.x : i == 1 ? x.y : i == 2 ? x.z : x.w);
    }
    __device__ __forceinline__ static uint4 pack(const float *f)
    {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

// UB-byte units as the low words of a uint4 (the rest zero): read-only
// loads, coherent loads (the residual, which may be written in place), stores.
template <int UB>
__device__ __forceinline__ uint4 ld_unit_nc(const void *p)
{
    if (UB == 16)
        return ld_nc_v4(p);
    uint32_t a, b;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(a), "=r"(b) : "l"(p));
    return make_uint4(a, b, 0u, 0u);
}
template <int UB>
__device__ __forceinline__ uint4 ld_unit(const void *p)
{
    if (UB == 16) {
        uint4 v;
        asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                     : "l"(p)
                     : "memory");
        return v;
    }
    uint32_t a, b;
    asm volatile("ld.global.v2.u32 {%0,%1}, [%2];" : "=r"(a), "=r"(b) : "l"(p) : "memory");
    return make_uint4(a, b, 0u, 0u);
}
template <int UB>
__device__ __forceinline__ void st_unit(void *p, const uint4 &x)
{
    if (UB == 16)
        st_v4(p, x);
    else
        st_v2u32(p, x.x, x.y);
}

__device__ __forceinline__ uint4 ld_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

// ------------------------------------------- cluster exchange (DSMEM + mbarrier)
__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
// the same shared-memory offset in cluster CTA `rank`, as a shared::cluster address
// CTAs in this CTA's thread-block cluster (1 when launched without clusters)
__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t n;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
    return n;
}

// The fused kernels address the shared memory of the other CTAs of their
// cluster, so a grid launched without the cluster shape it was planned for
// (as a profiler replaying the launch did) must not run: every CTA records
// SFAR_ERR_UNSUPPORTED and leaves at once.
__device__ __forceinline__ bool wrong_cluster_shape(SfarCtl *ctl, int CL, int rank, int cta)
{
    if (cluster_size() == (uint32_t)CL)
        return false;
    if (threadIdx.x == 0)
        sfar_record_code(ctl, SFAR_ERR_UNSUPPORTED, rank, cta, -1, 0, SFAR_WAIT_CLUSTER);
    return true;
}

__device__ __forceinline__ uint32_t map_cta(uint32_t addr, uint32_t rank)
{
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}
__device__ __forceinline__ void mbar_init(uint32_t mb, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(mb), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init_cluster()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mb, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mb), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t mb, uint32_t parity)
{
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done)
                 : "r"(mb), "r"(parity)
                 : "memory");
    return done != 0;
}
__device__ __forceinline__ void st_async_u32(uint32_t raddr, uint32_t v, uint32_t rmbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(raddr), "r"(v),
                 "r"(rmbar)
                 : "memory");
}
__device__ __forceinline__ void st_async_u64(uint32_t raddr, unsigned long long v, uint32_t rmbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b64 [%0], %1, [%2];" ::"r"(raddr), "l"(v),
                 "r"(rmbar)
                 : "memory");
}
__device__ __forceinline__ void st_async_v4u32(uint32_t raddr, uint4 v, uint32_t rmbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(raddr),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(rmbar)
                 : "memory");
}
__device__ __forceinline__ void st_async_v2u64(uint32_t raddr, unsigned long long a, unsigned long long b,
                                               uint32_t rmbar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b64 [%0], {%1, %2}, [%3];" ::"r"(raddr),
                 "l"(a), "l"(b), "r"(rmbar)
                 : "memory");
}
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Wait for one phase of a local mbarrier that the cluster's CTAs complete.
// Every CTA of the cluster sends its statistics on every path, after waits
// that are each bounded by at most twice the handle's limit, so this wait
// does not give up when another CTA records a failure (which would let this
// CTA exit while a peer's store into its shared memory is still coming); it
// gives up only after 8 times the limit, records a fault and returns false.
__device__ __forceinline__ bool cluster_mbar_wait(uint32_t mb, uint32_t parity, SfarCtl *ctl, int r, int k,
                                                  uint32_t e)
{
    unsigned long long t0 = 0;
    uint32_t it = 0;
    while (!mbar_try_wait_cluster(mb, parity)) {
        if ((++it & 127u) != 0)
            continue;
        const unsigned long long now = globaltimer();
        if (t0 == 0) {
            t0 = now;
        } else if (now - t0 > (ld_relaxed_u64(&ctl->timeout_ns) << 3)) {
            sfar_record_fault(ctl, r, k, -1, e, SFAR_WAIT_CLUSTER);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const uint32_t lo = __shfl_xor_sync(SFAR_FULL, (uint32_t)x, o);
        const uint32_t hi = __shfl_xor_sync(SFAR_FULL, (uint32_t)(x >> 32), o);
        x += ((unsigned long long)hi << 32) | lo;
    }
    return x;
}

}  // namespace
