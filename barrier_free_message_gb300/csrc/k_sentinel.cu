// k_sentinel.cu -- one-shot AllReduce over sentinel-prefilled receive buffers.
//
// "Every Microsecond Counts" (page 1), section "Four barrier-free
// mechanisms", part 2 (sentinel): the receive buffer is prefilled with a NaN
// pattern that real data never takes; the reader polls the data itself until
// it differs from the pattern, so no flag is sent and the full bandwidth
// carries payload.  The buffer must be refilled with the pattern before it is
// used again, and data equal to the pattern would never be accepted (here:
// the bounded wait gives up and reports it).  The refill is resetRange of the
// page's API (section "Unified primitives and API design").
//
// Sentinel: all-ones bits (bf16 0xffff, fp32 0xffffffff), a negative NaN
// with every payload bit set; finite sums and the workloads' inputs never
// produce it.  A unit is accepted when none of its elements equals the
// sentinel; each 4-byte word is single-copy atomic, so an element is never
// seen half-written.
//
// Units (UB): a thread carries UB bytes (8, or 16) of input, stored raw at
// bytes [UB v, UB v + UB) of every peer's slot: one 8-byte store, poll and
// refill per peer, with twice the threads of 16-byte units.
//
// Reset ordering: the reader refills exactly the slots it consumed, in its
// own buffer (parity e & 1), before its epoch e + 1 sends (kernel boundary,
// or the overlap-mode release of `done`).  A peer writes that parity again
// only at epoch e + 2, after it has received this rank's epoch e + 1 data,
// so the refill happens before the rewrite.
#include "sfar_units.cuh"

template <int DT>
__device__ __forceinline__ bool has_sentinel(uint4 x)
{
    if (DT == 1)
        return x.x == 0xffffffffu || x.y == 0xffffffffu || x.z == 0xffffffffu || x.w == 0xffffffffu;
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    bool s = false;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        s |= (w[i] & 0xffffu) == 0xffffu || (w[i] >> 16) == 0xffffu;
    return s;
}

// one unit of the receive region: raw UB bytes
template <int UB>
__device__ __forceinline__ uint4 ld_slot(const uint8_t *p)
{
    if (UB == 16)
        return ld_relaxed_v4(p);
    const unsigned long long w = ld_relaxed_u64(reinterpret_cast<const unsigned long long *>(p));
    return make_uint4((uint32_t)w, (uint32_t)(w >> 32), 0u, 0u);
}
template <int UB>
__device__ __forceinline__ void st_slot(uint8_t *p, const uint4 &x)
{
    if (UB == 16)
        st_relaxed_v4(p, x);
    else
        st_relaxed_u64(p, (unsigned long long)x.x | ((unsigned long long)x.y << 32));
}

template <int DT, int RB, bool TEST, int UB>
__global__ void __launch_bounds__(SFAR_THREADS) k_sentinel(const __grid_constant__ SfarArgs a)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    const int R = a.R, K = a.K;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    const unsigned long long nbytes = a.n * ES;
    const unsigned long long nvec = (nbytes + UB - 1ull) / UB;
    const unsigned long long stride = (unsigned long long)K * blockDim.x;
    const unsigned long long v0 = (unsigned long long)k * blockDim.x + threadIdx.x;
    if (v0 * UB < nbytes)
        prefetch_l2((const char *)a.in[r] + v0 * UB);
    const SfarEntry ent = sfar_entry<true>(a);     // early ticket (see sfar_entry)
    const uint4 x0 = load_unit<ES, UB>(a.in[r], v0, nbytes);     // before the prologue's barrier
    SfarCall c;
    if (!sfar_prologue<TEST>(a, r, k, c, ent))
        return;
    const uint32_t e = c.e;
    const size_t slot = a.slot;
    sfar_stamp_after(c, TP_INPUT, x0.x);

    if (!c.drop) {
        for (unsigned long long v = v0; v < nvec; v += stride) {
            const uint4 x = v == v0 ? x0 : load_unit<ES, UB>(a.in[r], v, nbytes);
#pragma unroll
            for (int i = 0; i < RB - 1; ++i) {
                if (i < R - 1) {
                    const int p = peer_of(r, i);
                    st_slot<UB>(a.region + ((size_t)(p * 2 + c.par) * R + r) * slot + v * UB, x);
                }
            }
        }
    }

    sfar_stamp(c, TP_SENT);
    sfar_mid_delay<TEST>(c);
    uint8_t *mine = a.region + (size_t)(r * 2 + c.par) * R * slot;
    const uint4 sent = make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu);
    bool ok = true;
    for (unsigned long long v = v0; v < nvec && ok; v += stride) {
        const uint4 own = v == v0 ? x0 : load_unit<ES, UB>(a.in[r], v, nbytes);
        // every round re-reads all peers still holding the sentinel at once
        uint4 x[RB];
        bool rdy[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) {
            rdy[q] = q >= R || q == r;
            if (!rdy[q])
                x[q] = ld_slot<UB>(mine + (size_t)q * slot + v * UB);
        }
        SfarWaiter w;
        while (true) {
            bool all = true;
#pragma unroll
            for (int q = 0; q < RB; ++q) {
                if (!rdy[q])
                    rdy[q] = !has_sentinel<DT>(x[q]);
                all = all && rdy[q];
            }
            if (all)
                break;
#pragma unroll
            for (int q = 0; q < RB; ++q)
                if (!rdy[q])
                    x[q] = ld_slot<UB>(mine + (size_t)q * slot + v * UB);
            if (w.tick(a.ctl)) {
                int late = -1;
#pragma unroll
                for (int q = RB - 1; q >= 0; --q)
                    if (!rdy[q])
                        late = q;
                sfar_record_fault(a.ctl, r, k, late, e, SFAR_WAIT_SENTINEL);
                ok = false;
                break;
            }
        }
        if (!ok)
            break;
        SfarAcc<DT> acc;
        acc.set(r == 0 ? own : x[0]);
#pragma unroll
        for (int q = 1; q < RB; ++q)
            if (q < R)
                acc.add(q == r ? own : x[q]);
        store_unit<ES, UB>(a.out[r], v, nbytes, acc.get());
        // refill the consumed slots with the sentinel
#pragma unroll
        for (int q = 0; q < RB; ++q)
            if (q < R && q != r)
                st_slot<UB>(mine + (size_t)q * slot + v * UB, sent);
    }
    sfar_stamp(c, TP_RECEIVED);
    sfar_epilogue(a, r, k, e);
    sfar_stamp(c, TP_EXIT);
}

const void *sfar_kernel_sentinel(int dt, int wide, int test)
{
#define SFAR_PICK(D, W, T)                                        \
    if (dt == D && wide == W && test == T)                       \
        return (const void *)k_sentinel<D, (W ? 16 : 8), (T != 0), SFAR_SENT_UNIT>;
    SFAR_PICK(0, 0, 0) SFAR_PICK(0, 0, 1) SFAR_PICK(0, 1, 0) SFAR_PICK(0, 1, 1)
    SFAR_PICK(1, 0, 0) SFAR_PICK(1, 0, 1) SFAR_PICK(1, 1, 0) SFAR_PICK(1, 1, 1)
#undef SFAR_PICK
    return nullptr;
}
