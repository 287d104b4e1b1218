// k_atomic.cu -- two-shot AllReduce by hardware atomic accumulation into
// 128-byte lines that carry their own arrival counter.
//
// "Every Microsecond Counts" (page 1), section "Four barrier-free
// mechanisms", part 4 (the LL128 atomic algorithm), and the table of variants
// in section "Unified primitives and API design" (two-phase LL128): a
// reduce-scatter then an all-gather.  The data are cut into 128-byte lines
// whose first 4 bytes are a counter; every rank adds its part of a line into
// the owner's copy with hardware atomic adds and then increments the line's
// counter; the owner polls the counter locally, and once it equals the
// number of ranks the line holds the complete sum.
//
// Line layout (both phases): word 0 = counter (reduce-scatter) or epoch flag
// (all-gather), words 1..31 = 31 consecutive elements.  Reduce-scatter words
// are binary32 accumulators for either element type (the pages fix no
// precision for the accumulation; binary32 is the precision of every other
// protocol's fold); all-gather words carry the rounded result bits.
//
// Determinism: the atomics add in whatever order the L2 performs them, so
// this protocol alone is NOT bit-exact with the rank-order fold.  Each atomic
// binary32 add rounds to nearest even and flushes subnormal operands and
// results to zero, so before the final rounding the accumulator differs from
// the exact sum by at most 2 (R - 1) 2^-24 sum_q |x_q| + 2 R 2^-126 (the
// classical bound for recursive summation in any order, doubled to cover its
// second-order term, plus one flushed subnormal per operand and per result).
// Sums whose partial sums are all exact (e.g. small integers) are exact in
// every order and therefore bit-exact.
//
// Chunks: owner p holds elements [p*c, min(n, (p+1)*c)), c = ceil(n / R)
// rounded up to whole lines (31 elements).  Regions: accumulators
// [owner][parity][line], all-gather lines [receiver][parity][owner][line].
// CTA (r, k), warp w handles line indices k*W + w + j*K*W of every chunk, one
// line per warp step, lane i on word i.
//   1. Every rank adds each of its valid elements into the owners' lines
//      (all R owners, itself included), fences once per warp, then adds 1 to
//      each of those lines' counters.
//   2. Owner r waits for counter == R on all of a warp's lines at once, then
//      line by line reads the sums, rounds them once, writes its own output
//      and every peer's all-gather line, and clears the accumulator line (data
//      and counter) for the next use of this parity; then fences and sets the
//      all-gather flags to e.
//   3. Every rank polls the all-gather flags of every (owner, line) pair of
//      the warp at once and copies the results to its output.
// Reuse: a line of parity e & 1 is added to again at epoch e + 2.  A rank
// starts epoch e + 2 only after it finished epoch e + 1, which needed every
// owner's epoch e + 1 all-gather lines, which each owner sends only after
// finishing epoch e, clearing included (serial launches add the kernel
// boundary on top).  So the clearing never races with the next adds, and the
// counter target is R for every call whatever the message size.
#include "sfar_prims.cuh"

__device__ __forceinline__ void red_add_f32(float *p, float v)
{
    asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void red_add_u32(uint32_t *p, uint32_t v)
{
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A counter increment with release semantics: it heads a release sequence that
// every later increment of the counter continues, so the owner's acquire load
// that reads the count R synchronises with every contributor.
__device__ __forceinline__ void red_release_add_u32(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ float ld_relaxed_f32(const float *p)
{
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

// Element idx of a rank's input, widened to binary32 (read-only input).
template <int ES>
__device__ __forceinline__ float load_elem(const void *base, unsigned long long idx)
{
    if (ES == 2) {
        unsigned short b;
        asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(b) : "l"((const char *)base + idx * 2ull));
        return __uint_as_float((uint32_t)b << 16);
    }
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"((const char *)base + idx * 4ull));
    return v;
}

// binary32 -> result bits of the element type (one rounding to nearest even)
template <int ES>
__device__ __forceinline__ uint32_t round_elem(float v)
{
    if (ES == 2)
        return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
    return __float_as_uint(v);
}

template <int ES>
__device__ __forceinline__ void store_elem(void *base, unsigned long long idx, uint32_t bits)
{
    if (ES == 2)
        asm volatile("st.global.u16 [%0], %1;" ::"l"((char *)base + idx * 2ull), "h"((unsigned short)bits)
                     : "memory");
    else
        st_u32((char *)base + idx * 4ull, bits);
}

template <int DT, int RB, bool TEST>
__global__ void __launch_bounds__(SFAR_THREADS, 3) k_atomic(const __grid_constant__ SfarArgs a)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    const int R = a.R, K = a.K;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned long long n = a.n, c = a.chunk, L = c / 31ull;
    const unsigned long long it0 = (unsigned long long)k * (blockDim.x >> 5) + warp;
    const unsigned long long its = (unsigned long long)K * (blockDim.x >> 5);
    // element of owner p's line `it` on this lane (lane 0 holds the counter)
    auto elem = [&](int p, unsigned long long it) { return (unsigned long long)p * c + it * 31ull + lane - 1; };
    auto line_valid = [&](int p, unsigned long long it) { return it < L && (unsigned long long)p * c + it * 31ull < n; };

    // owners in the order this rank sends to them: r + 1, r + 2, ... (mod R),
    // so that the ranks start on different owners
    auto owner = [&](int j) { return (r + 1 + j) % R; };
    // this lane's first element for every owner, loaded ahead of the prologue
    // (the L2 prefetch may precede the programmatic-launch wait, the load not)
    float x0[RB];
#pragma unroll
    for (int j = 0; j < RB; ++j) {
        x0[j] = 0.f;
        if (j < R && lane >= 1 && it0 < L && elem(owner(j), it0) < n)
            prefetch_l2((const char *)a.in[r] + elem(owner(j), it0) * ES);
    }
    const SfarEntry ent = sfar_entry(a);
#pragma unroll
    for (int j = 0; j < RB; ++j)
        if (j < R && lane >= 1 && it0 < L && elem(owner(j), it0) < n)
            x0[j] = load_elem<ES>(a.in[r], elem(owner(j), it0));
    SfarCall cl;
    if (!sfar_prologue<TEST>(a, r, k, cl, ent))
        return;
    const uint32_t e = cl.e;
    sfar_stamp_after(cl, TP_INPUT, __float_as_uint(x0[0]));
    const size_t slot = a.slot;                     // bytes per (owner, parity) of either region
    float *acc = reinterpret_cast<float *>(a.region);
    uint8_t *ag = a.region2;
    auto acc_line = [&](int p, unsigned long long it) {
        return acc + ((size_t)(p * 2 + cl.par) * slot) / 4 + it * 32ull;
    };
    auto ag_line = [&](int q, int p, unsigned long long it) {
        return reinterpret_cast<uint32_t *>(ag + ((size_t)(q * 2 + cl.par) * R + p) * slot) + it * 32ull;
    };

    // 1. reduce-scatter: atomic adds, one fence, counters
    if (!cl.drop) {
        for (unsigned long long it = it0; it < L; it += its) {
#pragma unroll
            for (int j = 0; j < RB; ++j) {
                if (j < R) {
                    const int p = owner(j);
                    const unsigned long long idx = elem(p, it);
                    if (lane >= 1 && idx < n) {
                        const float v = it == it0 ? x0[j] : load_elem<ES>(a.in[r], idx);
                        red_add_f32(acc_line(p, it) + lane, v);
                    }
                }
            }
        }
        __syncwarp();                    // every lane's data reductions before the counter lanes' release
        for (unsigned long long it = it0; it < L; it += its)
            for (int p = lane; p < R; p += 32)
                if (line_valid(p, it))
                    red_release_add_u32(reinterpret_cast<uint32_t *>(acc_line(p, it)), 1u);
    }
    sfar_stamp(cl, TP_SENT);
    sfar_mid_delay<TEST>(cl);

    // 2. owner: wait for all R contributions of every line of this warp at
    // once (lane m polls the counter of the warp's line m, m + 32, ...), then
    // round, all-gather send and clear line by line
    bool ok = true;
    unsigned long long nl = 0;          // this warp's lines of owner r
    while (line_valid(r, it0 + nl * its))
        ++nl;
    {
        int lok = 1;
        for (unsigned long long m = lane; m < nl && lok; m += 32) {
            const uint32_t *cnt = reinterpret_cast<const uint32_t *>(acc_line(r, it0 + m * its));
            SfarWaiter w;
            while (ld_acquire_u32(cnt) != (uint32_t)R) {
                if (w.tick(a.ctl)) {
                    sfar_record_fault(a.ctl, r, k, -1, e, SFAR_WAIT_COUNTER);
                    lok = 0;
                    break;
                }
            }
        }
        ok = __all_sync(SFAR_FULL, lok) != 0;
        __syncwarp();                           // each lane's acquisition, passed on to the warp
    }
    for (unsigned long long m = 0; m < nl && ok; ++m) {
        const unsigned long long it = it0 + m * its;
        float *line = acc_line(r, it);
        const float s = lane >= 1 ? ld_relaxed_f32(line + lane) : 0.f;
        st_relaxed_u32(reinterpret_cast<uint32_t *>(line + lane), 0u);     // lane 0: the counter
        const uint32_t bits = round_elem<ES>(s);
        const unsigned long long idx = elem(r, it);
        if (lane >= 1 && idx < n) {
            store_elem<ES>(a.out[r], idx, bits);
            if (!cl.drop) {
#pragma unroll
                for (int i = 0; i < RB - 1; ++i)
                    if (i < R - 1)
                        st_u32(ag_line(peer_of(r, i), r, it) + lane, bits);
            }
        }
    }
    if (ok && !cl.drop) {
        __syncwarp();
        for (unsigned long long m = 0; m < nl; ++m)
            for (int i = lane; i < R - 1; i += 32)
                st_release_u32(ag_line(peer_of(r, i), r, it0 + m * its), e);
    }

    // 3. all-gather receive: the warp polls the flags of every (owner, line)
    // pair it will read at once (lane j takes pairs j, j + 32, ...), then
    // every owner's words of each line are read in one round and copied out
    unsigned long long na = 0;          // this warp's lines of the widest owner chunk
    while (it0 + na * its < L)
        ++na;
    if (ok) {
        int lok = 1;
        const unsigned long long pairs = na * (unsigned long long)(R - 1);
        for (unsigned long long q = lane; q < pairs && lok; q += 32) {
            const unsigned long long m = q / (unsigned long long)(R - 1);
            const int p = peer_of(r, (int)(q - m * (unsigned long long)(R - 1)));
            const unsigned long long it = it0 + m * its;
            if (!line_valid(p, it))
                continue;
            const uint32_t *f = ag_line(r, p, it);
            SfarWaiter w(true);
            while (ld_acquire_u32(f) != e) {
                if (w.tick(a.ctl)) {
                    sfar_record_fault(a.ctl, r, k, p, e, SFAR_WAIT_AG);
                    lok = 0;
                    break;
                }
            }
        }
        ok = __all_sync(SFAR_FULL, lok) != 0;
        __syncwarp();
    }
    for (unsigned long long m = 0; m < na && ok; ++m) {
        const unsigned long long it = it0 + m * its;
        uint32_t y[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q)
            if (q < R && q != r && lane >= 1 && elem(q, it) < n)
                y[q] = ld_relaxed_u32(ag_line(r, q, it) + lane);
#pragma unroll
        for (int q = 0; q < RB; ++q)
            if (q < R && q != r && lane >= 1 && elem(q, it) < n)
                store_elem<ES>(a.out[r], elem(q, it), y[q]);
    }
    sfar_stamp(cl, TP_RECEIVED);
    sfar_epilogue(a, r, k, e);
    sfar_stamp(cl, TP_EXIT);
}

const void *sfar_kernel_atomic(int dt, int wide, int test)
{
#define SFAR_PICK(D, W, T)                                        \
    if (dt == D && wide == W && test == T)                       \
        return (const void *)k_atomic<D, (W ? 16 : 8), (T != 0)>;
    SFAR_PICK(0, 0, 0) SFAR_PICK(0, 0, 1) SFAR_PICK(0, 1, 0) SFAR_PICK(0, 1, 1)
    SFAR_PICK(1, 0, 0) SFAR_PICK(1, 0, 1) SFAR_PICK(1, 1, 0) SFAR_PICK(1, 1, 1)
#undef SFAR_PICK
    return nullptr;
}
