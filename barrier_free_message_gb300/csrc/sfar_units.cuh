// sfar_units.cuh -- a rank's input and output in units of UB bytes (16, 8 or
// 4) per thread, for the one-shot kernels that give each thread one unit per
// round (LL, sentinel).  A unit is returned as the low words of a uint4, the
// rest zero; bytes past the message end read as zero and are not written,
// element by element.
#pragma once
#include "sfar_prims.cuh"

__device__ __forceinline__ void st_relaxed_u64(void *p, unsigned long long v)
{
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// UB (8 or 4) bytes of a rank's input
template <int ES, int UB>
__device__ __forceinline__ uint4 load_part(const void *base, unsigned long long v, unsigned long long nbytes)
{
    const unsigned long long off = v * (unsigned long long)UB;
    uint32_t w0 = 0, w1 = 0;
    const char *p = (const char *)base + off;
    if (off + UB <= nbytes) {
        if (UB == 8)
            asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(w0), "=r"(w1) : "l"(p));
        else
            asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(w0) : "l"(p));
    } else if (off < nbytes) {
        const int rem = (int)(nbytes - off);
        if (ES == 4) {
            w0 = *(const uint32_t *)p;
        } else {
            const uint16_t *q = (const uint16_t *)p;
            w0 = q[0];
            if (rem > 2) w0 |= (uint32_t)q[1] << 16;
            if (rem > 4) w1 = q[2];
        }
    }
    return make_uint4(w0, w1, 0u, 0u);
}

template <int ES, int UB>
__device__ __forceinline__ void store_part(void *base, unsigned long long v, unsigned long long nbytes, uint4 x)
{
    const unsigned long long off = v * (unsigned long long)UB;
    char *p = (char *)base + off;
    if (off + UB <= nbytes) {
        if (UB == 8)
            st_v2u32(p, x.x, x.y);
        else
            st_u32(p, x.x);
        return;
    }
    if (off >= nbytes)
        return;
    const int rem = (int)(nbytes - off);
    if (ES == 4) {
        *(uint32_t *)p = x.x;
    } else {
        uint16_t *q = (uint16_t *)p;
        q[0] = (uint16_t)x.x;
        if (rem > 2) q[1] = (uint16_t)(x.x >> 16);
        if (rem > 4) q[2] = (uint16_t)x.y;
    }
}

// unit v of a rank's input or output, any UB
template <int ES, int UB>
__device__ __forceinline__ uint4 load_unit(const void *base, unsigned long long v, unsigned long long nbytes)
{
    if (UB == 16)
        return load_vec<ES>(base, v, nbytes);
    return load_part<ES, UB == 16 ? 8 : UB>(base, v, nbytes);
}
template <int ES, int UB>
__device__ __forceinline__ void store_unit(void *base, unsigned long long v, unsigned long long nbytes, uint4 x)
{
    if (UB == 16)
        store_vec<ES>(base, v, nbytes, x);
    else
        store_part<ES, UB == 16 ? 8 : UB>(base, v, nbytes, x);
}
