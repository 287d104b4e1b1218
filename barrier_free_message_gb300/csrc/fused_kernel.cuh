// fused_kernel.cuh -- one-shot AllReduce over LL packets fused with the
// residual add and the RMS normalisation that follow it in a decode layer.
// The kernel template; k_fused.cu instantiates it with 16-byte units,
// k_fused8.cu with 8-byte units (two translation units built in parallel).
//
// "vLLM distributed inference core" (page 2), sections one and two: in the
// decode step the normalisation runs right after the AllReduce of the
// attention output and of the MLP down projection, on the compute stream,
// once the AllReduce is complete.  "Every Microsecond Counts" (page 1),
// section "Unified primitives and API design": the one-shot kernel reduces
// the received values in registers and writes the result; here the result
// does not go to memory but straight into the epilogue.
//
// What it computes per rank r and row i (h = hidden elements):
//   a = the AllReduce result, rounded to the element type T (bit for bit the
//       one-shot LL result);
//   z = T(a (+) res)                    binary32 add, one rounding;
//   ms = ldexp(float(S) (/) h, 2E - F), S = sum of z^2 in units of 2^(2E - F)
//       with each term truncated to a whole unit: E is the exponent of the
//       smallest power of two above every |z| of the row, F = 53 -
//       ceil(log2 h), so S is an exact integer below 2^53 -- the same for
//       every launch geometry and every order of the reduction; float(S) and
//       the division round once each in binary32; NaN in the row -> NaN,
//       else inf -> +inf;
//   rstd = 1 (/) sqrt(ms (+) eps), y = T((z (*) rstd) (*) w), each binary32
//       operation rounded to nearest even.
// Outputs: out[r] = y, res_out[r] = z (z is stored as soon as it is formed,
// before the row statistics).
//
// Units: a thread carries UB bytes of a row per unit: 16, or 8 (one LL line
// per peer instead of two, as the plain LL kernel) for an AllReduce of rows
// of up to 16 KB that gives every cluster at most one row.
//
// Layout: a row is spread over one thread-block cluster of CL CTAs; thread t
// of cluster CTA c holds in-row units c*T + t + j*CL*T (j < vpt), for B
// rows at a time (B = 1, or up to 4 when vpt = 1), whose statistics share
// each round.  The row
// statistics (the largest |z| as magnitude bits, then the integer S) are
// reduced within each warp, and every warp stores its partial into its slot
// in every cluster CTA's shared memory (st.async, distributed shared memory),
// which completes bytes on that CTA's mbarrier; each CTA then combines the
// slots itself.  Two such rounds per batch of rows; integer max and sum are
// associative, so the order does not matter.  The G clusters of a rank take
// rows g, g + G, ...; CTA (r, k), k = g*CL + c, is blockIdx r*K + k with
// K = G*CL, so the epoch ticket and the LL slots are those of the plain LL
// kernel (receive region [receiver][parity][sender][2 * S bytes]).
//
// Every CTA of a cluster sends its statistics on every path: a CTA that
// finds the handle failed, or a wait that gives up, only skips work.
#pragma once
#include "fused_common.cuh"

namespace {

// Receive vector v from every peer's LL packets (bounded polling, all late
// peers re-read at once) and fold in rank order with the rank's own vector.
template <int DT, int RB, int UB>
__device__ __forceinline__ uint4 ll_recv_fold(const SfarArgs &a, int r, int k, uint32_t e, int par,
                                              unsigned long long v, uint4 own, bool &ok)
{
    const int R = a.R;
    const uint8_t *mine = a.region + (size_t)(r * 2 + par) * R * a.slot;
    constexpr int W2 = UB == 16 ? RB : 1;
    unsigned long long w0[RB], w1[RB], w2[W2], w3[W2];
    bool rdy[RB];
#pragma unroll
    for (int q = 0; q < RB; ++q) {
        rdy[q] = q >= R || q == r;
        if (!rdy[q]) {
            const uint8_t *src = mine + (size_t)q * a.slot + v * 2ull * UB;
            ld_relaxed_v2u64(src, w0[q], w1[q]);
            if (UB == 16)
                ld_relaxed_v2u64(src + 16, w2[UB == 16 ? q : 0], w3[UB == 16 ? q : 0]);
        }
    }
    SfarWaiter w;
    while (true) {
        bool all = true;
#pragma unroll
        for (int q = 0; q < RB; ++q) {
            if (!rdy[q])
                rdy[q] = UB == 16 ? ll_ready(w0[q], w1[q], w2[UB == 16 ? q : 0], w3[UB == 16 ? q : 0], e)
                                  : ((uint32_t)(w0[q] >> 32) == e && (uint32_t)(w1[q] >> 32) == e);
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
            return make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < RB; ++q)
            if (!rdy[q]) {
                const uint8_t *src = mine + (size_t)q * a.slot + v * 2ull * UB;
                ld_relaxed_v2u64(src, w0[q], w1[q]);
                if (UB == 16)
                    ld_relaxed_v2u64(src + 16, w2[UB == 16 ? q : 0], w3[UB == 16 ? q : 0]);
            }
    }
    auto data = [&](int q) {
        if (UB == 16)
            return make_uint4((uint32_t)w0[q], (uint32_t)w1[q], (uint32_t)w2[UB == 16 ? q : 0],
                              (uint32_t)w3[UB == 16 ? q : 0]);
        return make_uint4((uint32_t)w0[q], (uint32_t)w1[q], 0u, 0u);
    };
    SfarAcc<DT> acc;
    acc.set(r == 0 ? own : data(0));
#pragma unroll
    for (int q = 1; q < RB; ++q)
        if (q < R)
            acc.add(q == r ? own : data(q));
    return acc.get();
}

}  // namespace

// Two CTAs per SM for 8-byte units and R <= 8 (at most 128 registers; the
// batched variant spills 12 bytes): twice the clusters per rank, so more rows
// take 8-byte units.  The wide variant keeps one (it would spill 290 bytes).
template <int DT, int RB, bool AR, bool TEST, int NB, int UB>
__global__ void __launch_bounds__(SFAR_NORM_THREADS, UB == 8 && RB <= 8 ? 2 : 1)
    k_fused(const __grid_constant__ SfarArgs a, const __grid_constant__ SfarNormArgs na)
{
    using V = Vec<DT>;
    constexpr int ES = DT == 0 ? 2 : 4;
    constexpr int NE = V::N * UB / 16;                   // elements per unit
    const int R = a.R, K = a.K, CL = na.CL, G = na.G;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    const int g = k / CL, cr = k - g * CL;      // 1-D clusters of CL consecutive CTAs: the rank in the cluster
    const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (wrong_cluster_shape(a.ctl, CL, r, k))
        return;
    const unsigned long long h = na.hidden, rows = na.rows;
    const unsigned long long VR = h * ES / (unsigned long long)UB;       // units per row
    const unsigned long long ustride = (unsigned long long)CL * T;
    const unsigned long long u0 = (unsigned long long)cr * T + tid;

    // one slot per (cluster CTA, warp): every warp sends its partial straight
    // to every cluster CTA
    constexpr int WMAX = SFAR_NORM_THREADS / 32;
    __shared__ __align__(16) unsigned long long s_sum[SFAR_NORM_CLMAX * WMAX][SFAR_NORM_VMAX];
    __shared__ __align__(16) uint4 s_max[SFAR_NORM_CLMAX * WMAX];
    __shared__ __align__(8) unsigned long long s_mbar[2];      // [0]: row maxima, [1]: row sums
    const uint32_t mb_max = smem_u32(&s_mbar[0]), mb_sum = smem_u32(&s_mbar[1]);
    const int W = T >> 5, nslots = CL * W, slot = cr * W + warp;

    // first input vector of the first row, loaded ahead of the prologue (the
    // L2 prefetch may precede the programmatic-launch wait, the load not)
    const bool has0 = (unsigned long long)g < rows && u0 < VR;
    const unsigned long long v00 = (unsigned long long)g * VR + u0;
    if (has0) {
        if (AR)
            prefetch_l2((const char *)a.in[r] + v00 * UB);
        prefetch_l2((const char *)na.res[r] + v00 * UB);
        prefetch_l2((const char *)na.weight + u0 * UB);
    }
    SfarCall c;
    c.e = 0;
    c.par = 0;
    c.drop = false;
    c.mid_delay_ns = 0;
    c.trace = nullptr;
    bool alive = true;
    uint4 x00 = make_uint4(0, 0, 0, 0), r00 = x00, w00 = x00;
    if (AR) {
        const SfarEntry ent = sfar_entry<true>(a);     // early ticket (see sfar_entry)
        if (has0)
            x00 = ld_unit_nc<UB>((const char *)a.in[r] + v00 * UB);
        alive = sfar_prologue<TEST>(a, r, k, c, ent);
    } else {
        pdl_wait();
    }
    // the first row's residual and weight of vector j = 0: loaded now, so
    // their latency overlaps the sends and the AllReduce round trip
    if (has0) {
        r00 = ld_unit<UB>((const char *)na.res[r] + v00 * UB);
        w00 = ld_unit_nc<UB>((const char *)na.weight + u0 * UB);
        if (!AR)
            x00 = ld_unit_nc<UB>((const char *)a.in[r] + v00 * UB);
    }
    const uint32_t e = c.e;
    bool ok = alive;

    // 1. AllReduce send: every vector of every row of this cluster, as LL
    // packets into every peer's slot r (the plain LL kernel's layout)
    if (AR && ok && !c.drop) {
        const unsigned long long eh = (unsigned long long)e << 32;
        for (unsigned long long i = g; i < rows; i += G) {
#pragma unroll
            for (int j = 0; j < SFAR_NORM_VMAX; ++j) {
                const unsigned long long u = u0 + j * ustride;
                if (u < VR) {
                    const unsigned long long v = i * VR + u;
                    const uint4 x = (i == (unsigned long long)g && j == 0) ? x00
                                                                            : ld_unit_nc<UB>((const char *)a.in[r] + v * UB);
                    const unsigned long long p0 = x.x | eh, p1 = x.y | eh, p2 = x.z | eh, p3 = x.w | eh;
#pragma unroll
                    for (int q = 0; q < RB - 1; ++q) {
                        if (q < R - 1) {
                            const int p = peer_of(r, q);
                            uint8_t *dst = a.region + ((size_t)(p * 2 + c.par) * R + r) * a.slot + v * 2ull * UB;
                            st_relaxed_v2u64(dst, p0, p1);
                            if (UB == 16)
                                st_relaxed_v2u64(dst + 16, p2, p3);
                        }
                    }
                }
            }
        }
    }
    if (AR) {
        sfar_stamp(c, TP_SENT);
        sfar_mid_delay<TEST>(c);
    }

    // Row statistics travel between the cluster's CTAs as st.async stores
    // into each other's shared memory, each completing bytes on the
    // receiver's mbarrier.  The mbarriers must be initialised before any peer
    // signals them: init, fence, cluster arrive here (after the sends,
    // which are more urgent); the matching wait comes
    // just before the first store to a peer.
    if (tid == 0) {
        mbar_init(mb_max, 1);
        mbar_init(mb_sum, 1);
        fence_mbar_init_cluster();
    }
    __syncthreads();
    cluster_arrive_relaxed();
    bool cluster_ready = false;
    uint32_t phase = 0;


    // 2. rows in batches of B: the AllReduce result, z, then the row
    // statistics of the whole batch in two cluster rounds (each warp sends its
    // B maxima, then its B sums), then y.  NB = 1: one row, slot q of a thread
    // is its vector q of the row; NB = 4 (one vector per row and thread): slot
    // q is row i0 + q*G.
    const int vpt = na.vpt, B = na.B;
    for (unsigned long long i0 = g; i0 < rows; i0 += (unsigned long long)G * B) {
        uint4 zv[SFAR_NORM_VMAX], wv[SFAR_NORM_VMAX], rv[SFAR_NORM_VMAX], xv[SFAR_NORM_VMAX];
        bool valid[SFAR_NORM_VMAX];
        unsigned long long vq[SFAR_NORM_VMAX];
        // independent loads first: residual, weight and own input of every slot
#pragma unroll
        for (int q = 0; q < SFAR_NORM_VMAX; ++q) {
            const int bq = NB == 1 ? 0 : q, j = NB == 1 ? q : 0;
            const unsigned long long i = i0 + (unsigned long long)bq * G, u = u0 + j * ustride;
            zv[q] = wv[q] = rv[q] = xv[q] = make_uint4(0, 0, 0, 0);
            valid[q] = bq < B && j < vpt && i < rows && u < VR;
            vq[q] = i * VR + u;
            if (valid[q]) {
                if (i == (unsigned long long)g && j == 0) {
                    rv[q] = r00;
                    wv[q] = w00;
                    xv[q] = x00;
                } else {
                    rv[q] = ld_unit<UB>((const char *)na.res[r] + vq[q] * UB);
                    wv[q] = ld_unit_nc<UB>((const char *)na.weight + u * UB);
                    xv[q] = ld_unit_nc<UB>((const char *)a.in[r] + vq[q] * UB);
                }
            }
        }
        uint32_t lmax[NB];                                        // per row of the batch
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
            lmax[bb] = 0u;
#pragma unroll
        for (int q = 0; q < SFAR_NORM_VMAX; ++q) {
            if (valid[q] && ok) {
                const uint4 av = AR ? ll_recv_fold<DT, RB, UB>(a, r, k, e, c.par, vq[q], xv[q], ok) : xv[q];
                float zf[V::N];
#pragma unroll
                for (int t = 0; t < V::N; ++t)
                    zf[t] = t < NE ? __fadd_rn(V::get(av, t), V::get(rv[q], t)) : 0.f;
                zv[q] = V::pack(zf);
                uint32_t m = 0;
                if (DT == 0) {
                    m = max_mag_bf16(zv[q], NE);
                } else {
#pragma unroll
                    for (int t = 0; t < NE; ++t)
                        m = max(m, mag_bits(V::get(zv[q], t)));
                }
                lmax[NB == 1 ? 0 : q] = max(lmax[NB == 1 ? 0 : q], m);
                if (ok)
                    st_unit<UB>((char *)na.res_out[r] + vq[q] * UB, zv[q]);    // z is final: stored now
            }
        }
        if (i0 == (unsigned long long)g)
            sfar_stamp(c, TP_INPUT);          // first batch: AllReduce result and z in registers
        // row maxima of the magnitude bits: each warp's B maxima go to its slot
        // in every cluster CTA
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
            if (bb < B)
                lmax[bb] = __reduce_max_sync(SFAR_FULL, lmax[bb]);
        if (!cluster_ready) {
            cluster_wait();                    // every peer's mbarriers are initialised
            cluster_ready = true;
        }
        if (tid == 0)
            mbar_arrive_expect_tx(mb_max, (uint32_t)nslots * (NB == 1 ? 4u : 16u));
        if (lane < CL) {
            if (NB == 1)
                st_async_u32(map_cta(smem_u32(&s_max[slot]), lane), lmax[0], map_cta(mb_max, lane));
            else
                st_async_v4u32(map_cta(smem_u32(&s_max[slot]), lane),
                               make_uint4(lmax[0], lmax[NB > 1 ? 1 : 0], lmax[NB > 2 ? 2 : 0], lmax[NB > 3 ? 3 : 0]),
                               map_cta(mb_max, lane));
        }
        if (!cluster_mbar_wait(mb_max, phase, a.ctl, r, k, e))
            ok = false;
        uint32_t M[NB];
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
            M[bb] = 0u;
        // the lanes share the slots, then the warp combines them (a maximum and,
        // below, an integer sum: the same bits in any order).  Measured against
        // every lane reading every slot (up to 64): the decode row (R = 8, one
        // row of 8192 bf16) 5.46 -> 5.06 us per call.
        for (int qs = lane; qs < nslots; qs += 32) {
            const uint4 m4 = s_max[qs];
            M[0] = max(M[0], m4.x);
            if (NB > 1) {
                M[NB > 1 ? 1 : 0] = max(M[NB > 1 ? 1 : 0], m4.y);
                M[NB > 2 ? 2 : 0] = max(M[NB > 2 ? 2 : 0], m4.z);
                M[NB > 3 ? 3 : 0] = max(M[NB > 3 ? 3 : 0], m4.w);
            }
        }
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
            M[bb] = __reduce_max_sync(SFAR_FULL, M[bb]);
        // the truncated squares of each row, summed as integers
        unsigned long long lsum[NB];
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
            lsum[bb] = 0ull;
#pragma unroll
        for (int q = 0; q < SFAR_NORM_VMAX; ++q) {
            const int bq = NB == 1 ? 0 : q;
            if (valid[q] && M[bq] != 0 && M[bq] < 0x7f800000u) {
                const int E = exp_above(M[bq]);
                if (DT == 0) {
                    const SqScale sc = sq_scale(E, na.F);
#pragma unroll
                    for (int t = 0; t < NE; ++t)
                        lsum[bq] += sq_term_narrow(V::get(zv[q], t), sc);
                } else {
#pragma unroll
                    for (int t = 0; t < NE; ++t)
                        lsum[bq] += sq_term(V::get(zv[q], t), E, na.F);
                }
            }
        }
#pragma unroll
        for (int bb = 0; bb < NB; ++bb)
            if (bb < B)
                lsum[bb] = warp_sum_u64(lsum[bb]);
        if (tid == 0)
            mbar_arrive_expect_tx(mb_sum, (uint32_t)nslots * (NB == 1 ? 8u : 32u));
        if (lane < CL) {
            if (NB == 1) {
                st_async_u64(map_cta(smem_u32(&s_sum[slot][0]), lane), lsum[0], map_cta(mb_sum, lane));
            } else {
                st_async_v2u64(map_cta(smem_u32(&s_sum[slot][0]), lane), lsum[0], lsum[NB > 1 ? 1 : 0],
                               map_cta(mb_sum, lane));
                st_async_v2u64(map_cta(smem_u32(&s_sum[slot][2]), lane), lsum[NB > 2 ? 2 : 0], lsum[NB > 3 ? 3 : 0],
                               map_cta(mb_sum, lane));
            }
        }
        if (!cluster_mbar_wait(mb_sum, phase, a.ctl, r, k, e))
            ok = false;
        phase ^= 1u;
        float rstd[NB];
#pragma unroll
        for (int bb = 0; bb < NB; ++bb) {
            rstd[bb] = 0.f;
            if (bb >= B)
                continue;
            unsigned long long S = 0;
            for (int qs = lane; qs < nslots; qs += 32)
                S += s_sum[qs][bb];
            S = warp_sum_u64(S);
            const float ms = mean_square(M[bb], S, h, na.F);
            rstd[bb] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, na.eps)));
        }
        if (i0 == (unsigned long long)g)
            sfar_stamp(c, TP_RECEIVED);       // first batch: both cluster rounds done
#pragma unroll
        for (int q = 0; q < SFAR_NORM_VMAX; ++q) {
            if (valid[q] && ok) {
                const float rs = rstd[NB == 1 ? 0 : q];
                float yf[V::N];
#pragma unroll
                for (int t = 0; t < V::N; ++t)
                    yf[t] = t < NE ? __fmul_rn(__fmul_rn(V::get(zv[q], t), rs), V::get(wv[q], t)) : 0.f;
                st_unit<UB>((char *)a.out[r] + vq[q] * UB, V::pack(yf));
            }
        }
    }
    // A CTA leaves only after its last statistics wait, so every store that a
    // peer makes into its shared memory has landed (the mbarrier counts the
    // bytes); the cluster barrier opened at the start is closed first.
    if (!cluster_ready)
        cluster_wait();
    if (AR && alive) {
        sfar_epilogue(a, r, k, e);
        sfar_stamp(c, TP_EXIT);
    }
}

// The instantiation table of one unit size.
#define SFAR_FUSED_TABLE(NAME, UNIT)                                                                       \
    const void *NAME(int dt, int wide, int allreduce, int test, int batch)                               \
    {                                                                                                     \
        if (!allreduce)                                                                                   \
            wide = test = 0; /* the normalisation alone neither receives nor reads knobs */               \
        const int nb = batch > 1 ? 4 : 1;                                                                 \
        SFAR_FUSED_PICK_NB(0, 0, 1, 0, UNIT) SFAR_FUSED_PICK_NB(0, 0, 1, 1, UNIT)                         \
        SFAR_FUSED_PICK_NB(0, 1, 1, 0, UNIT) SFAR_FUSED_PICK_NB(0, 1, 1, 1, UNIT)                         \
        SFAR_FUSED_PICK_NB(1, 0, 1, 0, UNIT) SFAR_FUSED_PICK_NB(1, 0, 1, 1, UNIT)                         \
        SFAR_FUSED_PICK_NB(1, 1, 1, 0, UNIT) SFAR_FUSED_PICK_NB(1, 1, 1, 1, UNIT)                         \
        SFAR_FUSED_PICK_NB(0, 0, 0, 0, UNIT) SFAR_FUSED_PICK_NB(1, 0, 0, 0, UNIT)                         \
        return nullptr;                                                                                   \
    }
#define SFAR_FUSED_PICK(D, W, A, T, N, U)                                                                 \
    if (dt == D && wide == W && allreduce == A && test == T && nb == N)                                  \
        return (const void *)k_fused<D, (W ? 16 : 8), (A != 0), (T != 0), N, U>;
#define SFAR_FUSED_PICK_NB(D, W, A, T, U) SFAR_FUSED_PICK(D, W, A, T, 1, U) SFAR_FUSED_PICK(D, W, A, T, 4, U)
