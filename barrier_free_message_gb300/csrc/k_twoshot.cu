// k_twoshot.cu -- two-shot AllReduce (reduce-scatter, then all-gather) over
// LL128 lines with double-buffered epochs, for medium messages.
//
// "Every Microsecond Counts" (page 1), section "Unified primitives and API
// design", table of variants: the two-shot LLBuffer variant (double
// buffering, 64 KB to 1 MB) and the two-phase LL128 variant; section "Four
// barrier-free mechanisms", part 4: reduce-scatter then all-gather over
// 128-byte lines with a flag per line.  "SiFAR" (page 3), section "Limits of
// existing algorithms": each rank owns one chunk, reduces it, and broadcasts
// the reduced chunk.
//
// Chunks: owner j holds elements [j*c, min(n, (j+1)*c)); c is ceil(n / R)
// rounded up to a whole warp iteration (4 lines = 496 payload bytes) so that
// every chunk starts on a line group.  Chunking does not change any element's
// fold.  Regions: RS [owner][parity][sender][lines], AG
// [receiver][parity][owner][lines].  CTA (r, k), warp w handles iterations
// k*8 + w + j*K*8 of every chunk, so each exchange is between the CTAs of
// index k of two ranks.
//   1. RS send: rank r's slice of every other chunk j -> owner j's slot r.
//   2. Owner r polls its R - 1 slots, folds in rank order 0..R-1 (its own
//      slice at position r), rounds once, writes the result to its own output
//      and to every peer's AG slot r.
//   3. Every rank polls the AG slots of the other owners and unpacks them.
// Double buffering: parity e & 1; the argument of the one-shot kernels holds
// for both regions because every CTA finishes all three phases of epoch e
// before any of its epoch e + 1 sends.
#include "sfar_lineflags.cuh"

template <int DT, int RB, bool TEST>
__global__ void __launch_bounds__(SFAR_THREADS) k_twoshot(const __grid_constant__ SfarArgs a)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    const SfarEntry ent = sfar_entry<true>(a);     // early ticket (see sfar_entry)
    const int R = a.R, K = a.K;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    SfarCall c;
    if (!sfar_prologue<TEST>(a, r, k, c, ent))
        return;
    const uint32_t e = c.e;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 3, m = lane & 7;
    const unsigned long long nbytes = a.n * ES;
    const unsigned long long cvec = a.chunk * ES / 16ull;       // vectors per chunk (multiple of 31)
    const unsigned long long nitc = cvec / 31ull;              // iterations per chunk
    const unsigned long long it0 = (unsigned long long)k * (blockDim.x >> 5) + warp;
    const unsigned long long its = (unsigned long long)K * (blockDim.x >> 5);
    const size_t slot = a.slot;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    uint8_t *rs = a.region, *ag = a.region2;

    // 1. reduce-scatter send: per line group, every peer's input vector is
    // loaded before the first store, so the R - 1 loads are in flight together
    if (!c.drop) {
        for (unsigned long long it = it0; it < nitc; it += its) {
            uint4 xs[RB - 1];
#pragma unroll
            for (int i = 0; i < RB - 1; ++i)
                if (i < R - 1)
                    xs[i] = lane < 31 ? load_vec<ES>(a.in[r], peer_of(r, i) * cvec + it * 31ull + lane, nbytes) : zero;
#pragma unroll
            for (int i = 0; i < RB - 1; ++i) {
                if (i < R - 1) {
                    const int j = peer_of(r, i);
                    uint8_t *dst = rs + ((size_t)(j * 2 + c.par) * R + r) * slot;
                    ll128_store_data(dst + (it * 4ull + g) * 128ull, m, ll128_pack(xs[i], lane));
                }
            }
        }
        // the warp barrier orders every lane's payload stores before the flag
        // lanes' release stores (one flag per lane and peer)
        __syncwarp();
        for (unsigned long long it = it0; it < nitc; it += its)
            for (int i = m; i < R - 1; i += 8) {
                const int j = peer_of(r, i);
                st_release_u32((uint32_t *)(rs + ((size_t)(j * 2 + c.par) * R + r) * slot + (it * 4ull + g) * 128ull),
                               e);
            }
    }

    sfar_stamp(c, TP_SENT);
    sfar_mid_delay<TEST>(c);

    // 2. owner: receive, reduce, all-gather send
    const uint8_t *rs_mine = rs + (size_t)(r * 2 + c.par) * R * slot;
    bool ok = true;
    for (unsigned long long it = it0; it < nitc; it += its) {
        const size_t loff = (it * 4ull + g) * 128ull;
        const int lok = wait_line_flags<RB>(rs_mine, slot, loff, r, R, m, e, a.ctl, k, SFAR_WAIT_RS, false) ? 1 : 0;
        ok = __all_sync(SFAR_FULL, lok) != 0;
        if (!ok)
            break;
        __syncwarp();                   // each lane's acquisition, passed on to the warp
        const unsigned long long vb = r * cvec + it * 31ull + lane;
        const uint4 x = lane < 31 ? load_vec<ES>(a.in[r], vb, nbytes) : zero;
        const uint4 own = ll128_pack(x, lane);
        uint4 y[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q)
            if (q < R && q != r)
                y[q] = ld_relaxed_v4(rs_mine + (size_t)q * slot + loff + 16 * m);
        SfarAcc<DT> acc;
        acc.set(r == 0 ? own : y[0]);
#pragma unroll
        for (int q = 1; q < RB; ++q)
            if (q < R)
                acc.add(q == r ? own : y[q]);
        const uint4 res = acc.get();
        if (!c.drop) {
#pragma unroll
            for (int i = 0; i < RB - 1; ++i)
                if (i < R - 1) {
                    const int p = peer_of(r, i);
                    ll128_store_data(ag + ((size_t)(p * 2 + c.par) * R + r) * slot + loff, m, res);
                }
        }
        const uint4 o = ll128_unpack(res, lane);
        if (lane < 31)
            store_vec<ES>(a.out[r], vb, nbytes, o);
    }
    if (ok && !c.drop) {
        __syncwarp();
        for (unsigned long long it = it0; it < nitc; it += its)
            for (int i = m; i < R - 1; i += 8) {
                const int p = peer_of(r, i);
                st_release_u32((uint32_t *)(ag + ((size_t)(p * 2 + c.par) * R + r) * slot + (it * 4ull + g) * 128ull),
                               e);
            }
    }

    // 3. all-gather receive: lane (g, m) polls line g of owner peer m (and
    // m + 8), so all owners are waited for at once; then every owner's line
    // is read in one round and unpacked into this rank's output
    const uint8_t *ag_mine = ag + (size_t)(r * 2 + c.par) * R * slot;
    for (unsigned long long it = it0; it < nitc && ok; it += its) {
        const size_t loff = (it * 4ull + g) * 128ull;
        const int lok = wait_line_flags<RB>(ag_mine, slot, loff, r, R, m, e, a.ctl, k, SFAR_WAIT_AG, true) ? 1 : 0;
        ok = __all_sync(SFAR_FULL, lok) != 0;
        if (!ok)
            break;
        __syncwarp();
        uint4 y[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q)
            if (q < R && q != r)
                y[q] = ld_relaxed_v4(ag_mine + (size_t)q * slot + loff + 16 * m);
#pragma unroll
        for (int q = 0; q < RB; ++q) {
            if (q < R && q != r) {
                const uint4 o = ll128_unpack(y[q], lane);
                if (lane < 31)
                    store_vec<ES>(a.out[r], q * cvec + it * 31ull + lane, nbytes, o);
            }
        }
    }
    sfar_stamp(c, TP_RECEIVED);
    sfar_epilogue(a, r, k, e);
    sfar_stamp(c, TP_EXIT);
}

const void *sfar_kernel_twoshot(int dt, int wide, int test)
{
#define SFAR_PICK(D, W, T)                                        \
    if (dt == D && wide == W && test == T)                       \
        return (const void *)k_twoshot<D, (W ? 16 : 8), (T != 0)>;
    SFAR_PICK(0, 0, 0) SFAR_PICK(0, 0, 1) SFAR_PICK(0, 1, 0) SFAR_PICK(0, 1, 1)
    SFAR_PICK(1, 0, 0) SFAR_PICK(1, 0, 1) SFAR_PICK(1, 1, 0) SFAR_PICK(1, 1, 1)
#undef SFAR_PICK
    return nullptr;
}
