// k_twoshot_sent.cu -- two-shot AllReduce over sentinel-prefilled receive
// buffers, double buffered: the pages' algorithm for medium messages.
//
// "Every Microsecond Counts" (page 1), section "Unified primitives and API
// design", table of variants: the two-phase LLBuffer algorithm synchronises
// by sentinel with double buffering and serves 64 KB to 1 MB.  Section "Four
// barrier-free mechanisms", part 2 (sentinel: the reader polls the data
// itself until it differs from a NaN pattern that real data never takes, so
// every byte on the wire is payload; the buffer is refilled before reuse)
// and part 3 (double buffering: a received message is the licence to reuse
// the previous buffer).  "SiFAR" (page 3), section "Limits of existing
// algorithms": each rank owns one chunk, reduces it over all ranks
// (reduce-scatter) and hands the reduced chunk to every rank (all-gather).
//
// Chunks: owner j holds elements [j*c, min(n, (j+1)*c)); c is ceil(n / R)
// rounded up to 16 bytes.  A chunk moves in units of UB = 8 bytes; unit u of
// every chunk belongs to thread u mod T of CTA (u / T) mod K of every rank
// (T threads per CTA, K CTAs per rank), so each exchange is between the
// CTAs of one index k of two ranks.
// Units wholly past the end of the message are skipped by every side.
// Regions (prefilled with the sentinel): RS [owner][parity][sender][c bytes],
// AG [receiver][parity][owner][c bytes].
//   1. RS send: rank r stores its unit u of every other chunk j raw into
//      owner j's RS slot r.
//   2. Owner r polls the R - 1 RS slots of unit u at once until none holds
//      the sentinel, folds in rank order 0..R-1 (its own input at position
//      r), rounds once, refills the RS slots, stores the result into every
//      peer's AG slot r and into its own output.
//   3. Every rank polls the AG slots of unit u of all other owners at once,
//      stores them into its output and refills them.
// Two CTAs of 256 threads fit an SM (at most 128 registers: without the
// bound the R > 8 bf16 variant took 210 and one CTA per SM).
// Sentinel: all-ones bits (bf16 0xffff, fp32 0xffffffff).  Inputs must not
// contain it (a unit holding it is never accepted and the bounded wait
// reports a timeout); a reduced result never equals it: rounding a finite
// sum gives a number or an infinity, and a NaN produced by an addition is
// the canonical positive NaN.
// Reuse: a rank writes parity e & 1 of a peer's RS or AG region again only
// at epoch e + 2, and it does so after it has received data of epoch e + 1
// that the peer sent after finishing epoch e, refills included (kernel
// boundary, or the overlap-mode release of `done`).
#include "sfar_units.cuh"

#define TS_UB 8

namespace {

template <int DT>
__device__ __forceinline__ bool unit_has_sentinel(unsigned long long w)
{
    if (DT == 1)
        return (uint32_t)w == 0xffffffffu || (uint32_t)(w >> 32) == 0xffffffffu;
    return (w & 0xffffull) == 0xffffull || ((w >> 16) & 0xffffull) == 0xffffull ||
           ((w >> 32) & 0xffffull) == 0xffffull || (w >> 48) == 0xffffull;
}

__device__ __forceinline__ unsigned long long ld_unit(const uint8_t *p)
{
    return ld_relaxed_u64(reinterpret_cast<const unsigned long long *>(p));
}

__device__ __forceinline__ uint4 as_vec(unsigned long long w)
{
    return make_uint4((uint32_t)w, (uint32_t)(w >> 32), 0u, 0u);
}

__device__ __forceinline__ unsigned long long as_word(const uint4 &x)
{
    return (unsigned long long)x.x | ((unsigned long long)x.y << 32);
}

}  // namespace

template <int DT, int RB, bool TEST>
__global__ void __launch_bounds__(SFAR_THREADS, 2) k_twoshot_sent(const __grid_constant__ SfarArgs a)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    constexpr unsigned long long SENT = ~0ull;
    const int R = a.R, K = a.K;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    const unsigned long long nbytes = a.n * ES;
    const unsigned long long cbytes = a.chunk * ES;                 // bytes per chunk (multiple of 16)
    const unsigned long long cu = cbytes / TS_UB;                   // units per chunk
    const unsigned long long stride = (unsigned long long)K * blockDim.x;
    const unsigned long long u0 = (unsigned long long)k * blockDim.x + threadIdx.x;
    // unit u of chunk j is part of the message when its first byte is
    const auto valid = [&](int j, unsigned long long u) { return j * cbytes + u * TS_UB < nbytes; };
    const auto in_unit = [&](int j, unsigned long long u) {
        return load_part<ES, TS_UB>(a.in[r], (j * cbytes) / TS_UB + u, nbytes);
    };
    const SfarEntry ent = sfar_entry<true>(a);     // early ticket (see sfar_entry)
    SfarCall c;
    if (!sfar_prologue<TEST>(a, r, k, c, ent))
        return;
    const uint32_t e = c.e;
    const size_t slot = a.slot;
    uint8_t *rs = a.region, *ag = a.region2;

    // 1. reduce-scatter send: every peer's unit is loaded before the first
    // store, so the R - 1 loads are in flight together
    if (!c.drop) {
        for (unsigned long long u = u0; u < cu; u += stride) {
            unsigned long long xs[RB - 1];
#pragma unroll
            for (int i = 0; i < RB - 1; ++i)
                if (i < R - 1)
                    xs[i] = as_word(in_unit(peer_of(r, i), u));
#pragma unroll
            for (int i = 0; i < RB - 1; ++i) {
                if (i < R - 1) {
                    const int j = peer_of(r, i);
                    if (valid(j, u))
                        st_relaxed_u64(rs + ((size_t)(j * 2 + c.par) * R + r) * slot + u * TS_UB, xs[i]);
                }
            }
        }
    }
    sfar_stamp(c, TP_SENT);
    sfar_mid_delay<TEST>(c);

    // 2. owner: receive, fold, refill, all-gather send
    uint8_t *rs_mine = rs + (size_t)(r * 2 + c.par) * R * slot;
    bool ok = true;
    for (unsigned long long u = u0; u < cu && ok; u += stride) {
        if (!valid(r, u))
            break;                                       // later units of this chunk are past the end too
        const uint4 own = in_unit(r, u);
        unsigned long long x[RB];
        bool rdy[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) {
            rdy[q] = q >= R || q == r;
            if (!rdy[q])
                x[q] = ld_unit(rs_mine + (size_t)q * slot + u * TS_UB);
        }
        SfarWaiter w;
        while (true) {
            bool all = true;
#pragma unroll
            for (int q = 0; q < RB; ++q) {
                if (!rdy[q])
                    rdy[q] = !unit_has_sentinel<DT>(x[q]);
                all = all && rdy[q];
            }
            if (all)
                break;
#pragma unroll
            for (int q = 0; q < RB; ++q)
                if (!rdy[q])
                    x[q] = ld_unit(rs_mine + (size_t)q * slot + u * TS_UB);
            if (w.tick(a.ctl)) {
                int late = -1;
#pragma unroll
                for (int q = RB - 1; q >= 0; --q)
                    if (!rdy[q])
                        late = q;
                sfar_record_fault(a.ctl, r, k, late, e, SFAR_WAIT_RS);
                ok = false;
                break;
            }
        }
        if (!ok)
            break;
        SfarAcc<DT> acc;
        acc.set(r == 0 ? own : as_vec(x[0]));
#pragma unroll
        for (int q = 1; q < RB; ++q)
            if (q < R)
                acc.add(q == r ? own : as_vec(x[q]));
        const uint4 res = acc.get();
#pragma unroll
        for (int q = 0; q < RB; ++q)
            if (q < R && q != r)
                st_relaxed_u64(rs_mine + (size_t)q * slot + u * TS_UB, SENT);
        if (!c.drop) {
            const unsigned long long wres = as_word(res);
#pragma unroll
            for (int i = 0; i < RB - 1; ++i)
                if (i < R - 1) {
                    const int p = peer_of(r, i);
                    st_relaxed_u64(ag + ((size_t)(p * 2 + c.par) * R + r) * slot + u * TS_UB, wres);
                }
        }
        store_part<ES, TS_UB>(a.out[r], (r * cbytes) / TS_UB + u, nbytes, res);
    }

    // 3. all-gather receive: every other owner's unit u at once
    uint8_t *ag_mine = ag + (size_t)(r * 2 + c.par) * R * slot;
    for (unsigned long long u = u0; u < cu && ok; u += stride) {
        unsigned long long x[RB];
        bool rdy[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) {
            rdy[q] = q >= R || q == r || !valid(q, u);
            if (!rdy[q])
                x[q] = ld_unit(ag_mine + (size_t)q * slot + u * TS_UB);
        }
        SfarWaiter w(true);
        while (true) {
            bool all = true;
#pragma unroll
            for (int q = 0; q < RB; ++q) {
                if (!rdy[q]) {
                    rdy[q] = !unit_has_sentinel<DT>(x[q]);
                    if (rdy[q]) {
                        store_part<ES, TS_UB>(a.out[r], (q * cbytes) / TS_UB + u, nbytes, as_vec(x[q]));
                        st_relaxed_u64(ag_mine + (size_t)q * slot + u * TS_UB, SENT);
                    }
                }
                all = all && rdy[q];
            }
            if (all)
                break;
#pragma unroll
            for (int q = 0; q < RB; ++q)
                if (!rdy[q])
                    x[q] = ld_unit(ag_mine + (size_t)q * slot + u * TS_UB);
            if (w.tick(a.ctl)) {
                int late = -1;
#pragma unroll
                for (int q = RB - 1; q >= 0; --q)
                    if (!rdy[q])
                        late = q;
                sfar_record_fault(a.ctl, r, k, late, e, SFAR_WAIT_AG);
                ok = false;
                break;
            }
        }
    }
    sfar_stamp(c, TP_RECEIVED);
    sfar_epilogue(a, r, k, e);
    sfar_stamp(c, TP_EXIT);
}

const void *sfar_kernel_twoshot_sent(int dt, int wide, int test)
{
#define SFAR_PICK(D, W, T)                                          \
    if (dt == D && wide == W && test == T)                         \
        return (const void *)k_twoshot_sent<D, (W ? 16 : 8), (T != 0)>;
    SFAR_PICK(0, 0, 0) SFAR_PICK(0, 0, 1) SFAR_PICK(0, 1, 0) SFAR_PICK(0, 1, 1)
    SFAR_PICK(1, 0, 0) SFAR_PICK(1, 0, 1) SFAR_PICK(1, 1, 0) SFAR_PICK(1, 1, 1)
#undef SFAR_PICK
    return nullptr;
}
