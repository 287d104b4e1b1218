// k_ll.cu -- one-shot AllReduce over LL packets.
//
// "Every Microsecond Counts" (page 1), section "Four barrier-free
// mechanisms", part 1 (LL): data and flag travel together in one atomic
// write, the receiver polls the flag half, and half of every slot is flag, so
// payload efficiency is 50%.  Section "Unified primitives and API design": the
// one-shot kernel has each thread read its local value, broadcast it to the
// peers, receive-and-reduce everyone's value, write the result and advance
// the epoch.  No barrier of any kind.
//
// Layout: receive region [receiver][parity][sender][2 * S bytes]; input
// vector v (16 bytes) of sender q lands at bytes [32v, 32v + 32) of slot q as
// two LL lines {w0,e,w1,e} {w2,e,w3,e}, written as 8-byte words (each word is
// single-copy atomic, so flag == e proves its data word arrived).
// Grid: R * K CTAs of T threads; CTA (r, k) = blockIdx r * K + k handles
// vectors k*T + t + j*K*T of rank r.  Parity e & 1 double-buffers the
// region: a sender can reach parity e & 1 again only at epoch e + 2, and its
// CTA (r, k) of epoch e + 1 first received epoch e + 1 data from every peer's
// CTA k, which each peer sends only after finishing epoch e (section part 3:
// a received message is the licence to overwrite the previous buffer).
//
// Latency: the first input vector is loaded before the prologue's barrier,
// so its DRAM latency overlaps the epoch ticket; every poll round re-reads
// all peers that are not ready yet at once, so one round trip covers them all.
//
// Units (UB, 8 bytes for every rank count): a thread carries UB bytes of
// input, one 16-byte LL line {w0,e,w1,e} per peer at bytes [16v, 16v + 16)
// of the slot for UB = 8 (two lines for UB = 16, one 8-byte word {w0,e} for
// UB = 4).  Holding R - 1 peers' packets then takes half the registers of
// 16-byte units, with twice the threads.
#include "sfar_units.cuh"

// The packets of one unit from every peer: UB / 4 words {data, epoch}.
template <int RB, int UB>
struct LLSlots {
    static constexpr int NW = UB / 4;
    unsigned long long w[NW][RB];
    __device__ __forceinline__ void load(int q, const uint8_t *src)
    {
        if (NW == 1) {
            w[0][q] = ld_relaxed_u64(reinterpret_cast<const unsigned long long *>(src));
        } else {
            ld_relaxed_v2u64(src, w[0][q], w[NW > 1 ? 1 : 0][q]);
            if (NW == 4)
                ld_relaxed_v2u64(src + 16, w[NW > 2 ? 2 : 0][q], w[NW > 3 ? 3 : 0][q]);
        }
    }
    __device__ __forceinline__ bool ready(int q, uint32_t e) const
    {
        bool r = true;
#pragma unroll
        for (int i = 0; i < NW; ++i)
            r = r && (uint32_t)(w[i][q] >> 32) == e;
        return r;
    }
    __device__ __forceinline__ uint4 data(int q) const
    {
        return make_uint4((uint32_t)w[0][q], NW > 1 ? (uint32_t)w[NW > 1 ? 1 : 0][q] : 0u,
                          NW > 2 ? (uint32_t)w[NW > 2 ? 2 : 0][q] : 0u, NW > 3 ? (uint32_t)w[NW > 3 ? 3 : 0][q] : 0u);
    }
};

template <int DT, int RB, bool TEST, int UB>
__global__ void __launch_bounds__(SFAR_THREADS) k_ll(const __grid_constant__ SfarArgs a)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    const int R = a.R, K = a.K;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    const unsigned long long nbytes = a.n * ES;
    const unsigned long long nvec = (nbytes + UB - 1ull) / UB;
    const unsigned long long stride = (unsigned long long)K * blockDim.x;
    const unsigned long long v0 = (unsigned long long)k * blockDim.x + threadIdx.x;
    auto load_in = [&](unsigned long long v) { return load_unit<ES, UB>(a.in[r], v, nbytes); };
    if (v0 * UB < nbytes)
        prefetch_l2((const char *)a.in[r] + v0 * UB);
    const SfarEntry ent = sfar_entry(a);
    const uint4 x0 = load_in(v0);                         // zero past the end
    SfarCall c;
    if (!sfar_prologue<TEST>(a, r, k, c, ent))
        return;
    const uint32_t e = c.e;
    const unsigned long long eh = (unsigned long long)e << 32;
    const size_t slot = a.slot;
    sfar_stamp_after(c, TP_INPUT, x0.x);

    // send: pack each input vector once, store it into every peer's slot r
    if (!c.drop) {
        for (unsigned long long v = v0; v < nvec; v += stride) {
            const uint4 x = v == v0 ? x0 : load_in(v);
            const unsigned long long p0 = x.x | eh, p1 = x.y | eh, p2 = x.z | eh, p3 = x.w | eh;
#pragma unroll
            for (int i = 0; i < RB - 1; ++i) {
                if (i < R - 1) {
                    const int p = peer_of(r, i);
                    uint8_t *dst = a.region + ((size_t)(p * 2 + c.par) * R + r) * slot + v * 2ull * UB;
                    if (UB == 4) {
                        st_relaxed_u64(dst, p0);
                    } else {
                        st_relaxed_v2u64(dst, p0, p1);
                        if (UB == 16)
                            st_relaxed_v2u64(dst + 16, p2, p3);
                    }
                }
            }
        }
    }
    sfar_stamp(c, TP_SENT);
    sfar_mid_delay<TEST>(c);

    // receive and reduce: poll every peer's packets, fold in rank order
    const uint8_t *mine = a.region + (size_t)(r * 2 + c.par) * R * slot;
    bool ok = true;
    for (unsigned long long v = v0; v < nvec && ok; v += stride) {
        const uint4 own = v == v0 ? x0 : load_in(v);
        LLSlots<RB, UB> s;
        bool rdy[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q) {
            rdy[q] = q >= R || q == r;
            if (!rdy[q])
                s.load(q, mine + (size_t)q * slot + v * 2ull * UB);
        }
        SfarWaiter w;
        while (true) {
            bool all = true;
#pragma unroll
            for (int q = 0; q < RB; ++q) {
                if (!rdy[q])
                    rdy[q] = s.ready(q, e);
                all = all && rdy[q];
            }
            if (all)
                break;
            if (w.tick(a.ctl)) {
                int late = -1;
#pragma unroll
                for (int q = RB - 1; q >= 0; --q)
                    if (!rdy[q])
                        late = q;
                sfar_record_fault(a.ctl, r, k, late, e, SFAR_WAIT_LL);
                ok = false;
                break;
            }
#pragma unroll
            for (int q = 0; q < RB; ++q)
                if (!rdy[q])
                    s.load(q, mine + (size_t)q * slot + v * 2ull * UB);
        }
        if (!ok)
            break;
        SfarAcc<DT> acc;
        acc.set(r == 0 ? own : s.data(0));
#pragma unroll
        for (int q = 1; q < RB; ++q)
            if (q < R)
                acc.add(q == r ? own : s.data(q));
        store_unit<ES, UB>(a.out[r], v, nbytes, acc.get());
    }
    sfar_stamp(c, TP_RECEIVED);
    sfar_epilogue(a, r, k, e);
    sfar_stamp(c, TP_EXIT);
}

const void *sfar_kernel_ll(int dt, int wide, int test)
{
#define SFAR_PICK(D, W, T)                                   \
    if (dt == D && wide == W && test == T)                  \
        return (const void *)k_ll<D, (W ? 16 : 8), (T != 0), (W ? SFAR_LL_UNIT_WIDE : SFAR_LL_UNIT_NARROW)>;
    SFAR_PICK(0, 0, 0) SFAR_PICK(0, 0, 1) SFAR_PICK(0, 1, 0) SFAR_PICK(0, 1, 1)
    SFAR_PICK(1, 0, 0) SFAR_PICK(1, 0, 1) SFAR_PICK(1, 1, 0) SFAR_PICK(1, 1, 1)
#undef SFAR_PICK
    return nullptr;
}
