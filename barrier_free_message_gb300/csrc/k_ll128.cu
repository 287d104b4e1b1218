// k_ll128.cu -- one-shot AllReduce over LL128 lines.
//
// "Every Microsecond Counts" (page 1), section "Four barrier-free
// mechanisms", part 4 (LL128): data moves in 128-byte lines whose first
// 4 bytes are a counter/flag, and a reader polls the line's flag locally
// instead of waiting at a global barrier.  On the page the lines are
// accumulated by NVLink atomic adds; here each sender writes its own line
// (no floating-point atomics: their order would not be fixed) and the flag
// word carries the epoch.
//
// Line: word 0 = flag (epoch), words 1..31 = 124 bytes of payload.  A warp
// moves 4 lines (496 payload bytes = 31 input vectors) per iteration; lane
// l holds 16 bytes of line l / 8.  The writer stores the payload of all its
// lines, then __syncwarp (the warp barrier orders every lane's payload
// stores before what each lane does next), then the flag lanes store the
// epoch with st.release.gpu: the release covers the payload the flag lane
// has observed through the barrier.  The reader polls its flag with
// ld.acquire.gpu, then __syncwarp passes each lane's acquisition on to the
// lanes that read the other peers' payload of the same line.  The sum is
// folded in line layout (the reduction is element-wise and lines keep 4-byte
// words intact) and unpacked to vector layout for the output store.
//
// Layout: receive region [receiver][parity][sender][lines * 128 bytes];
// CTA (r, k), warp w handles iterations k*8 + w + j*K*8 of rank r's data.
#include "sfar_lineflags.cuh"

template <int DT, int RB, bool TEST>
__global__ void __launch_bounds__(SFAR_THREADS) k_ll128(const __grid_constant__ SfarArgs a)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    const SfarEntry ent = sfar_entry<true>(a);     // early ticket (see sfar_entry)
    const int R = a.R, K = a.K;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, g = lane >> 3, m = lane & 7;
    const unsigned long long nbytes = a.n * ES;
    const unsigned long long nvec = (nbytes + 15ull) >> 4;
    const unsigned long long nit = (nvec + 30ull) / 31ull;
    const unsigned long long it0 = (unsigned long long)k * (blockDim.x >> 5) + warp;
    const unsigned long long its = (unsigned long long)K * (blockDim.x >> 5);
    const uint4 zero = make_uint4(0, 0, 0, 0);
    // first group's input, loaded before the prologue's barrier
    const uint4 x0 = lane < 31 ? load_vec<ES>(a.in[r], it0 * 31ull + lane, nbytes) : zero;
    SfarCall c;
    if (!sfar_prologue<TEST>(a, r, k, c, ent))
        return;
    const uint32_t e = c.e;
    const size_t slot = a.slot;
    sfar_stamp_after(c, TP_INPUT, x0.x);

    // send: payload of every line to every peer, a warp barrier, then the flags
    if (!c.drop) {
        for (unsigned long long it = it0; it < nit; it += its) {
            const uint4 x = it == it0 ? x0 : (lane < 31 ? load_vec<ES>(a.in[r], it * 31ull + lane, nbytes) : zero);
            const uint4 y = ll128_pack(x, lane);
#pragma unroll
            for (int i = 0; i < RB - 1; ++i) {
                if (i < R - 1) {
                    const int p = peer_of(r, i);
                    uint8_t *line = a.region + ((size_t)(p * 2 + c.par) * R + r) * slot + (it * 4ull + g) * 128ull;
                    ll128_store_data(line, m, y);
                }
            }
        }
        __syncwarp();
        for (unsigned long long it = it0; it < nit; it += its)
            for (int i = m; i < R - 1; i += 8) {
                const int p = peer_of(r, i);
                st_release_u32((uint32_t *)(a.region + ((size_t)(p * 2 + c.par) * R + r) * slot +
                                            (it * 4ull + g) * 128ull),
                               e);
            }
    }

    sfar_stamp(c, TP_SENT);
    sfar_mid_delay<TEST>(c);

    // receive: poll the line flags, read the payload, fold in rank order
    const uint8_t *mine = a.region + (size_t)(r * 2 + c.par) * R * slot;
    bool ok = true;
    for (unsigned long long it = it0; it < nit; it += its) {
        const size_t loff = (it * 4ull + g) * 128ull;
        const int lok = wait_line_flags<RB>(mine, slot, loff, r, R, m, e, a.ctl, k, SFAR_WAIT_LL128, false) ? 1 : 0;
        ok = __all_sync(SFAR_FULL, lok) != 0;
        if (!ok)
            break;
        __syncwarp();                   // each lane's acquisition, passed on to the warp
        const uint4 x = it == it0 ? x0 : (lane < 31 ? load_vec<ES>(a.in[r], it * 31ull + lane, nbytes) : zero);
        const uint4 own = ll128_pack(x, lane);
        uint4 y[RB];
#pragma unroll
        for (int q = 0; q < RB; ++q)
            if (q < R && q != r)
                y[q] = ld_relaxed_v4(mine + (size_t)q * slot + loff + 16 * m);
        SfarAcc<DT> acc;
        acc.set(r == 0 ? own : y[0]);
#pragma unroll
        for (int q = 1; q < RB; ++q)
            if (q < R)
                acc.add(q == r ? own : y[q]);
        const uint4 res = ll128_unpack(acc.get(), lane);
        if (lane < 31)
            store_vec<ES>(a.out[r], it * 31ull + lane, nbytes, res);
    }
    sfar_stamp(c, TP_RECEIVED);
    sfar_epilogue(a, r, k, e);
    sfar_stamp(c, TP_EXIT);
}

const void *sfar_kernel_ll128(int dt, int wide, int test)
{
#define SFAR_PICK(D, W, T)                                      \
    if (dt == D && wide == W && test == T)                     \
        return (const void *)k_ll128<D, (W ? 16 : 8), (T != 0)>;
    SFAR_PICK(0, 0, 0) SFAR_PICK(0, 0, 1) SFAR_PICK(0, 1, 0) SFAR_PICK(0, 1, 1)
    SFAR_PICK(1, 0, 0) SFAR_PICK(1, 0, 1) SFAR_PICK(1, 1, 0) SFAR_PICK(1, 1, 1)
#undef SFAR_PICK
    return nullptr;
}
