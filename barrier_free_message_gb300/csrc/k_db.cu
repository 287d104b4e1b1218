// k_db.cu -- one-shot AllReduce with flags: the two-barrier baseline and its
// double-buffered variant.
//
// BASELINE ("Every Microsecond Counts" (page 1), section "Global memory
// barriers"; "SiFAR" (page 3), section "Limits of existing algorithms"):
// every rank writes its data into each peer's receive buffer, then a top
// barrier ("all writes done, wait for everyone before reading"), the reads
// and the reduction, then a bottom barrier ("all reads done, wait for
// everyone before the next round writes").  One receive buffer.
//
// DB ("SiFAR" (page 3), section "Technique 1"; page 1, section "Four
// barrier-free mechanisms", part 3): the same kernel with the receive buffers
// alternating by epoch parity, which makes the bottom barrier unnecessary;
// only the top barrier remains, here as one ready flag per (receiver, sender,
// CTA) written with release semantics after the data and polled with
// acquire semantics.
//
// A barrier between simulated ranks: CTA k of every rank stores epoch e into
// a flag of every peer, then polls its own R - 1 flags until they reach e.
// Flags only grow, so a waiter compares with >= and a fast peer that has
// already moved on to e + 1 still releases it.
//
// Layout: receive region [receiver][parity][sender][S bytes]; vector v at
// bytes [16v, 16v + 16) of its slot.  Flags fa (top) and fb (bottom) are
// [receiver][sender][CTA].
#include "sfar_prims.cuh"

// Store e into the peers' flags and wait for the peers' flags (warp 0 only).
// Returns false if a wait gave up.  The caller's __syncthreads before it
// orders every store (and, at the bottom barrier, every read) of the CTA
// before the storing lane's release; its __syncthreads after it passes each
// polling lane's acquisition on to the whole CTA.  (Against a warp-wide
// fence.acq_rel.gpu before the stores and after the polls, on GB300 at
// R = 8, 16 KB, graph-chained: DB 4.21 -> 3.88 us, BASELINE 5.95 -> 5.31 us
// per call.)
__device__ __forceinline__ bool flag_exchange(const SfarArgs &a, uint32_t *flags, int r, int k, uint32_t e,
                                              bool send, int where)
{
    const int lane = threadIdx.x & 31, R = a.R;
    if (send)
        for (int i = lane; i < R - 1; i += 32)
            st_release_u32(flags + sfar_flag((size_t)peer_of(r, i) * R + r, k), e);
    int ok = 1;
    for (int i = lane; i < R - 1 && ok; i += 32) {
        const int q = peer_of(r, i);
        const uint32_t *f = flags + sfar_flag((size_t)r * R + q, k);
        SfarWaiter w(where == SFAR_WAIT_BOTTOM);
        while (!epoch_ge(ld_acquire_u32(f), e))
            if (w.tick(a.ctl)) {
                sfar_record_fault(a.ctl, r, k, q, e, where);
                ok = 0;
                break;
            }
    }
    return __all_sync(SFAR_FULL, ok) != 0;
}

template <int DT, int RB, bool TEST, bool BASE>
__global__ void __launch_bounds__(SFAR_THREADS) k_db(const __grid_constant__ SfarArgs a)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    const int R = a.R, K = a.K;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    const unsigned long long nbytes = a.n * ES;
    const unsigned long long nvec = (nbytes + 15ull) >> 4;
    const unsigned long long stride = (unsigned long long)K * blockDim.x;
    const unsigned long long v0 = (unsigned long long)k * blockDim.x + threadIdx.x;
    if (v0 * 16ull < nbytes)
        prefetch_l2((const char *)a.in[r] + v0 * 16ull);
    const SfarEntry ent = sfar_entry<true>(a);     // early ticket (see sfar_entry)
    const uint4 x0 = load_vec<ES>(a.in[r], v0, nbytes);     // before the prologue's barrier
    SfarCall c;
    if (!sfar_prologue<TEST>(a, r, k, c, ent))
        return;
    const uint32_t e = c.e;
    const int par = BASE ? 0 : c.par;
    const size_t slot = a.slot;
    __shared__ int s_ok;
    sfar_stamp_after(c, TP_INPUT, x0.x);

    // send raw vectors
    if (!c.drop) {
        for (unsigned long long v = v0; v < nvec; v += stride) {
            const uint4 x = v == v0 ? x0 : load_vec<ES>(a.in[r], v, nbytes);
#pragma unroll
            for (int i = 0; i < RB - 1; ++i) {
                if (i < R - 1) {
                    const int p = peer_of(r, i);
                    st_v4(a.region + ((size_t)(p * 2 + par) * R + r) * slot + v * 16ull, x);
                }
            }
        }
    }
    __syncthreads();
    // top barrier / ready flags
    if (threadIdx.x < 32) {
        const bool ok = flag_exchange(a, a.fa, r, k, e, !c.drop, SFAR_WAIT_READY);
        if (threadIdx.x == 0)
            s_ok = ok;
    }
    __syncthreads();
    sfar_stamp(c, TP_SENT);      // here: after the top barrier
    // a slow reader (test knob): the data is there, its reads come late
    sfar_mid_delay<TEST>(c);

    if (s_ok) {
        const uint8_t *mine = a.region + (size_t)(r * 2 + par) * R * slot;
        for (unsigned long long v = v0; v < nvec; v += stride) {
            const uint4 own = v == v0 ? x0 : load_vec<ES>(a.in[r], v, nbytes);
            uint4 x[RB];
#pragma unroll
            for (int q = 0; q < RB; ++q)
                if (q < R && q != r)
                    x[q] = ld_relaxed_v4(mine + (size_t)q * slot + v * 16ull);
            SfarAcc<DT> acc;
            acc.set(r == 0 ? own : x[0]);
#pragma unroll
            for (int q = 1; q < RB; ++q)
                if (q < R)
                    acc.add(q == r ? own : x[q]);
            store_vec<ES>(a.out[r], v, nbytes, acc.get());
        }
        if (BASE) {
            // bottom barrier: nobody writes the next round before everyone read this one
            __syncthreads();
            if (threadIdx.x < 32)
                flag_exchange(a, a.fb, r, k, e, true, SFAR_WAIT_BOTTOM);
        }
    }
    sfar_stamp(c, TP_RECEIVED);
    sfar_epilogue(a, r, k, e);
    sfar_stamp(c, TP_EXIT);
}

const void *sfar_kernel_db(int dt, int wide, int test, int baseline)
{
#define SFAR_PICK(D, W, T, B)                                                  \
    if (dt == D && wide == W && test == T && baseline == B)                   \
        return (const void *)k_db<D, (W ? 16 : 8), (T != 0), (B != 0)>;
    SFAR_PICK(0, 0, 0, 0) SFAR_PICK(0, 0, 1, 0) SFAR_PICK(0, 1, 0, 0) SFAR_PICK(0, 1, 1, 0)
    SFAR_PICK(1, 0, 0, 0) SFAR_PICK(1, 0, 1, 0) SFAR_PICK(1, 1, 0, 0) SFAR_PICK(1, 1, 1, 0)
    SFAR_PICK(0, 0, 0, 1) SFAR_PICK(0, 0, 1, 1) SFAR_PICK(0, 1, 0, 1) SFAR_PICK(0, 1, 1, 1)
    SFAR_PICK(1, 0, 0, 1) SFAR_PICK(1, 0, 1, 1) SFAR_PICK(1, 1, 0, 1) SFAR_PICK(1, 1, 1, 1)
#undef SFAR_PICK
    return nullptr;
}
