// k_fused_ts.cu -- two-shot AllReduce fused with the residual add and the RMS
// normalisation, for calls of several rows.
//
// "SiFAR" (page 3), section "Limits of existing algorithms": in two-shot
// each rank owns a share of the message, reduces it over all ranks and hands
// the result to every rank, so no rank moves the whole message R times.
// "vLLM distributed inference core" (page 2), sections one and two: the
// normalisation runs right after the AllReduce of the attention output and
// of the MLP down projection.  Here the share is a row: its owner reduces the
// row once and normalises it for every rank, so the per-rank normalisation
// needs no second pass over the AllReduce result.
//
// What it computes is what the one-shot fused kernel (fused_kernel.cuh)
// computes, bit for bit: per rank p and row i,
//   a = the rank-order binary32 fold of every rank's row, rounded once;
//   z_p = T(a (+) res_p); ms_p from the exact integer sum of truncated
//   squares (fused_common.cuh); rstd_p = 1 (/) sqrt(ms_p (+) eps);
//   y_p = T((z_p (*) rstd_p) (*) w);  out[p] = y_p, res_out[p] = z_p.
//
// Ownership: the rows are dealt round-robin over the R*G clusters of the
// grid: cluster g of rank j (CTAs (j, g*CL) .. (j, g*CL + CL - 1)) owns rows
// i = j*G + g, + R*G, ...  Thread t of cluster CTA c holds unit c*T + t of
// the row (16 bytes; one unit per thread).  For each owned row a thread
//   1. reads its unit from every rank's input and folds them (R loads in
//      flight, with every rank's residual unit too for R <= 8);
//   2. forms z_p for every rank p and the largest |z_p| (R maxima per warp,
//      the first cluster exchange), then the truncated squares of every
//      z_p summed as integers (R sums per warp, the second exchange);
//   3. writes z_p into rank p's residual output as soon as it is formed, and
//      y_p into rank p's output after the statistics.
// The exchange is the one of the one-shot fused kernel: every warp stores its
// partials into its slot in every cluster CTA's shared memory (st.async,
// counted in bytes by that CTA's mbarrier); lane p of each warp then combines
// rank p's slots and hands the result to the warp by shuffle.  The R sums of
// a warp are reduced transposed (warp_sums_transposed), so the exchange costs
// a handful of shuffles rather than R full warp reductions.
//
// Synchronisation between simulated ranks (as the two-shot TMA kernel: the
// pages' counters reaching N, page 1 section "Four barrier-free mechanisms",
// part 4, kept as per-CTA epoch flags):
//   * arrival (top barrier): CTA (q, k) stores its epoch into arrive[q][k];
//     CTA (j, k) reads rank q's input and residual, and writes rank q's
//     outputs, only once arrive[q][k] holds this call's epoch;
//   * completion: after its stores, CTA (j, k) stores the epoch into
//     cmpl[p][j][k] for every rank p, and CTA (p, k) waits for every
//     owner (j, k) before it reports its call finished.
// Every CTA of the grid waits on others, so the host launches only grids
// whose clusters are all resident at once.  No receive buffers.  Every CTA
// of a cluster takes part in both exchange rounds of every owned row on every
// path: a CTA whose handle failed, or whose wait gave up, only skips work.
#include "fused_common.cuh"

// Largest magnitude (as binary32 magnitude bits) of the elements of one unit.
template <int DT>
__device__ __forceinline__ uint32_t unit_max(const uint4 &z)
{
    using V = Vec<DT>;
    if (DT == 0)
        return max_mag_bf16(z, V::N);
    uint32_t m = 0;
#pragma unroll
    for (int t = 0; t < V::N; ++t)
        m = max(m, mag_bits(V::get(z, t)));
    return m;
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long x, int m)
{
    const uint32_t lo = __shfl_xor_sync(SFAR_FULL, (uint32_t)x, m);
    const uint32_t hi = __shfl_xor_sync(SFAR_FULL, (uint32_t)(x >> 32), m);
    return ((unsigned long long)hi << 32) | lo;
}

// Warp sums of the RB (8 or 16) values of every lane, transposed: each xor
// step from 16 down keeps half of a lane's values and adds its partner's copy
// of them, until one value is left, and the last steps add it over the
// remaining lanes.  Lane l ends with the warp sum of value
// (l >> (5 - log2 RB)) & (RB - 1): log2(RB) + 1 ... 5 exchanges instead of
// RB * 5.
template <int RB>
__device__ __forceinline__ unsigned long long warp_sums_transposed(unsigned long long (&v)[RB], int lane)
{
    constexpr int LOG = RB == 16 ? 4 : 3;
#pragma unroll
    for (int s = 0; s < LOG; ++s) {
        const int n = RB >> (s + 1);
        const int off = 16 >> s;
        const bool up = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < RB / 2; ++j) {
            if (j < n) {
                const unsigned long long keep = up ? v[j + n] : v[j];
                const unsigned long long give = up ? v[j] : v[j + n];
                v[j] = keep + shfl_xor_u64(give, off);
            }
        }
    }
#pragma unroll
    for (int off = 16 >> LOG; off > 0; off >>= 1)
        v[0] += shfl_xor_u64(v[0], off);
    return v[0];
}

// Poll a flag of another rank until it reaches epoch e, with acquire loads;
// false if the bounded wait gave up.
__device__ __forceinline__ bool poll_acquire_ge(const uint32_t *f, uint32_t e, const SfarCtl *ctl, bool downstream)
{
    SfarWaiter w(downstream);
    while (!epoch_ge(ld_acquire_u32(f), e))
        if (w.tick(ctl))
            return false;
    return true;
}

template <int DT, int RB, bool TEST>
__global__ void __launch_bounds__(SFAR_NORM_THREADS, RB <= 8 ? 2 : 1)
    k_fused_ts(const __grid_constant__ SfarArgs a, const __grid_constant__ SfarNormArgs na)
{
    using V = Vec<DT>;
    constexpr int ES = DT == 0 ? 2 : 4;
    const int R = a.R, K = a.K, CL = na.CL, G = na.G;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    const int g = k / CL, cr = k - g * CL;      // 1-D clusters of CL consecutive CTAs
    const int T = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (wrong_cluster_shape(a.ctl, CL, r, k))
        return;
    const unsigned long long h = na.hidden, rows = na.rows;
    const unsigned long long VR = h * ES / 16ull;                 // units per row
    const unsigned long long u = (unsigned long long)cr * T + tid;
    const bool has_u = u < VR;
    const unsigned long long C = (unsigned long long)R * G;       // clusters of the grid
    const unsigned long long i0 = (unsigned long long)r * G + g;  // this cluster's first row

    constexpr int WMAX = SFAR_NORM_THREADS / 32;
    __shared__ __align__(16) uint32_t s_max[SFAR_NORM_CLMAX * WMAX][RB];
    __shared__ __align__(16) unsigned long long s_sum[SFAR_NORM_CLMAX * WMAX][RB];
    __shared__ __align__(8) unsigned long long s_mbar[2];      // [0]: row maxima, [1]: row sums
    __shared__ int s_ok;
    const uint32_t mb_max = smem_u32(&s_mbar[0]), mb_sum = smem_u32(&s_mbar[1]);
    const int W = T >> 5, nslots = CL * W, slot = cr * W + warp;
    const int R4 = (R + 3) >> 2;                  // 16-byte stores per slot in the first exchange

    const bool works = has_u && i0 < rows;
    if (works)
        prefetch_l2((const char *)na.weight + u * 16ull);
    const SfarEntry ent = sfar_entry<true>(a);     // early ticket (see sfar_entry)
    SfarCall c;
    c.e = 0;
    c.par = 0;
    c.drop = false;
    c.mid_delay_ns = 0;
    c.trace = nullptr;
    const bool alive = sfar_prologue<TEST>(a, r, k, c, ent);
    const uint32_t e = c.e;
    uint4 wv = make_uint4(0, 0, 0, 0);
    if (works)
        wv = ld_nc_v4((const char *)na.weight + u * 16ull);

    // arrival: this rank's input and residual are ready and its outputs free
    if (tid < 32) {
        if (tid == 0 && alive && !c.drop)
            st_release_u32(a.fa + sfar_pull_flag(r, k), e);
        int wok = alive ? 1 : 0;
        for (int i = lane; i < R - 1 && wok; i += 32) {
            const int q = peer_of(r, i);
            if (!poll_acquire_ge(a.fa + sfar_pull_flag(q, k), e, a.ctl, false)) {
                sfar_record_fault(a.ctl, r, k, q, e, SFAR_WAIT_ARRIVE);
                wok = 0;
            }
        }
        wok = __all_sync(SFAR_FULL, wok);     // the CTA barrier below passes the acquisitions on
        if (tid == 0)
            s_ok = wok;
    }
    // the exchange's mbarriers are initialised before any cluster peer
    // signals them: init, fence, cluster arrive here; the matching wait comes
    // before the first store to a peer
    if (tid == 0) {
        mbar_init(mb_max, 1);
        mbar_init(mb_sum, 1);
        fence_mbar_init_cluster();
    }
    __syncthreads();
    bool ok = s_ok != 0;
    cluster_arrive_relaxed();
    bool cluster_ready = false;
    uint32_t phase = 0;
    sfar_stamp(c, TP_SENT);
    sfar_mid_delay<TEST>(c);

    for (unsigned long long i = i0; i < rows; i += C) {
        const unsigned long long off = (i * VR + u) * 16ull;
        uint4 zs[RB];
        uint32_t lmax[RB];
#pragma unroll
        for (int p = 0; p < RB; ++p) {
            zs[p] = make_uint4(0, 0, 0, 0);
            lmax[p] = 0u;
        }
        if (ok && has_u) {
            // 1. the AllReduce of this unit: every rank's input, rank order
            uint4 xs[RB];
#pragma unroll
            for (int q = 0; q < RB; ++q)
                if (q < R)
                    xs[q] = ld_relaxed_v4((const char *)a.in[q] + off);
            if (RB <= 8) {
#pragma unroll
                for (int p = 0; p < RB; ++p)
                    if (p < R)
                        zs[p] = ld_relaxed_v4((const char *)na.res[p] + off);
            }
            SfarAcc<DT> acc;
            acc.set(xs[0]);
#pragma unroll
            for (int q = 1; q < RB; ++q)
                if (q < R)
                    acc.add(xs[q]);
            const uint4 av = acc.get();
            if (RB > 8) {
#pragma unroll
                for (int p = 0; p < RB; ++p)
                    if (p < R)
                        zs[p] = ld_relaxed_v4((const char *)na.res[p] + off);
            }
            // 2. z of every rank and its largest magnitude
#pragma unroll
            for (int p = 0; p < RB; ++p) {
                if (p < R) {
                    float zf[V::N];
#pragma unroll
                    for (int t = 0; t < V::N; ++t)
                        zf[t] = __fadd_rn(V::get(av, t), V::get(zs[p], t));
                    zs[p] = V::pack(zf);
                    lmax[p] = unit_max<DT>(zs[p]);
                    st_v4((char *)na.res_out[p] + off, zs[p]);     // z is final: stored now
                }
            }
        }
        if (i == i0)
            sfar_stamp(c, TP_INPUT);          // first row: AllReduce result and z in registers

        // first exchange: every warp's R maxima to its slot in every cluster CTA
#pragma unroll
        for (int p = 0; p < RB; ++p)
            if (p < R)
                lmax[p] = __reduce_max_sync(SFAR_FULL, lmax[p]);
        if (!cluster_ready) {
            cluster_wait();                    // every peer's mbarriers are initialised
            cluster_ready = true;
        }
        if (tid == 0)
            mbar_arrive_expect_tx(mb_max, (uint32_t)(nslots * R4 * 16));
        if (lane < CL) {
#pragma unroll
            for (int b = 0; b < RB / 4; ++b)
                if (b < R4)
                    st_async_v4u32(map_cta(smem_u32(&s_max[slot][4 * b]), lane),
                                   make_uint4(lmax[4 * b], lmax[4 * b + 1], lmax[4 * b + 2], lmax[4 * b + 3]),
                                   map_cta(mb_max, lane));
        }
        if (!cluster_mbar_wait(mb_max, phase, a.ctl, r, k, e))
            ok = false;
        // lane p combines rank p's maxima; every lane gets them all
        uint32_t mine = 0;
        if (lane < R)
            for (int qs = 0; qs < nslots; ++qs)
                mine = max(mine, s_max[qs][lane]);
        uint32_t M[RB];
#pragma unroll
        for (int p = 0; p < RB; ++p)
            M[p] = __shfl_sync(SFAR_FULL, mine, p);

        // second exchange: the truncated squares of every rank's row, summed as integers
        unsigned long long lsum[RB];
#pragma unroll
        for (int p = 0; p < RB; ++p) {
            lsum[p] = 0ull;
            if (p < R && M[p] != 0 && M[p] < 0x7f800000u) {
                const int E = exp_above(M[p]);
                if (DT == 0) {
                    const SqScale sc = sq_scale(E, na.F);
#pragma unroll
                    for (int t = 0; t < V::N; ++t)
                        lsum[p] += sq_term_narrow(V::get(zs[p], t), sc);
                } else {
#pragma unroll
                    for (int t = 0; t < V::N; ++t)
                        lsum[p] += sq_term(V::get(zs[p], t), E, na.F);
                }
            }
        }
        // lane l holds the warp sum of rank (l >> SH) & (RB - 1); the 2^SH lanes
        // holding rank p's sum send it to cluster CTAs c, c + 2^SH, ...
        constexpr int SH = RB == 16 ? 1 : 2;
        const unsigned long long wsum = warp_sums_transposed<RB>(lsum, lane);
        const int psum = (lane >> SH) & (RB - 1);
        if (tid == 0)
            mbar_arrive_expect_tx(mb_sum, (uint32_t)(nslots * R * 8));
        if (psum < R)
            for (int dst = lane & ((1 << SH) - 1); dst < CL; dst += 1 << SH)
                st_async_u64(map_cta(smem_u32(&s_sum[slot][psum]), dst), wsum, map_cta(mb_sum, dst));
        if (!cluster_mbar_wait(mb_sum, phase, a.ctl, r, k, e))
            ok = false;
        phase ^= 1u;
        float rs_mine = 0.f;
        if (lane < R) {
            unsigned long long S = 0;
            for (int qs = 0; qs < nslots; ++qs)
                S += s_sum[qs][lane];
            const float ms = mean_square(mine, S, h, na.F);
            rs_mine = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, na.eps)));
        }
        if (i == i0)
            sfar_stamp(c, TP_RECEIVED);       // first row: both cluster rounds done

        // 3. y and z of every rank
#pragma unroll
        for (int p = 0; p < RB; ++p) {
            const float rs = __shfl_sync(SFAR_FULL, rs_mine, p);
            if (p < R && ok && has_u) {
                float yf[V::N];
#pragma unroll
                for (int t = 0; t < V::N; ++t)
                    yf[t] = __fmul_rn(__fmul_rn(V::get(zs[p], t), rs), V::get(wv, t));
                st_v4((char *)a.out[p] + off, V::pack(yf));
            }
        }
    }
    // A CTA leaves only after its last statistics wait, so every store that a
    // peer makes into its shared memory has landed; the cluster barrier opened
    // at the start is closed first.
    if (!cluster_ready)
        cluster_wait();

    // completion: every rank learns that this owner's part of its rows is
    // written (release stores after the CTA barrier that orders the CTA's
    // output stores; acquire polls, passed on by the epilogue's barrier)
    __syncthreads();
    if (tid < 32) {
        if (ok && !c.drop)
            for (int p = lane; p < R; p += 32)
                if (p != r)
                    st_release_u32(a.fb + sfar_pull_flag((size_t)p * R + r, k), e);
        int wok = ok ? 1 : 0;
        for (int i = lane; i < R - 1 && wok; i += 32) {
            const int q = peer_of(r, i);
            if (!poll_acquire_ge(a.fb + sfar_pull_flag((size_t)r * R + q, k), e, a.ctl, true)) {
                sfar_record_fault(a.ctl, r, k, q, e, SFAR_WAIT_COMPLETE);
                wok = 0;
            }
        }
        __syncwarp();
    }
    if (alive) {
        sfar_epilogue(a, r, k, e);
        sfar_stamp(c, TP_EXIT);
    }
}

const void *sfar_kernel_fused_ts(int dt, int wide, int test)
{
#define SFAR_PICK(D, W, T)                                 \
    if (dt == D && wide == W && test == T)                \
        return (const void *)k_fused_ts<D, (W ? 16 : 8), (T != 0)>;
    SFAR_PICK(0, 0, 0) SFAR_PICK(0, 0, 1) SFAR_PICK(0, 1, 0) SFAR_PICK(0, 1, 1)
    SFAR_PICK(1, 0, 0) SFAR_PICK(1, 0, 1) SFAR_PICK(1, 1, 0) SFAR_PICK(1, 1, 1)
#undef SFAR_PICK
    return nullptr;
}
