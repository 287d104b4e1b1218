// k_tma.cu -- two-shot AllReduce for large messages with TMA bulk copies.
//
// "SiFAR" (page 3), section "Limits of existing algorithms": in two-shot
// each rank owns one chunk, reduces it over all ranks (reduce-scatter) and
// hands the reduced chunk to every rank (all-gather).  "Every Microsecond
// Counts" (page 1), section "Tensor parallelism and AllReduce": for large
// messages bandwidth, not latency, decides.  So this path moves the minimum
// bytes: owner j reads its chunk of every rank's input once and writes the
// reduced chunk once into every rank's output, with no staging buffers.
//
// Owner CTA (j, k) takes a contiguous range of chunk j and streams it in
// tiles through a ring of shared-memory stages, with the work split by warp:
//   * the producer warp: lane q issues the 1-D bulk copy of rank q's tile
//     (global -> shared, completion counted in bytes on the stage's "full"
//     mbarrier), after the stage's "empty" mbarrier says it was consumed;
//   * eight consumer warps: fold the R tiles from shared memory in rank
//     order, round once, write the tile into one of three output buffers
//     (after its "free" mbarrier), then arrive on the stage's "empty" and the
//     buffer's "full" mbarriers;
//   * the store warp: lane p issues the bulk copy shared -> global into rank
//     p's output, and frees a buffer once the copies reading it are done.
// No CTA-wide barrier in the steady state; every mbarrier wait is bounded.
// A CTA in which a wait gave up lets every copy it issued land before it
// leaves, so no copy writes into shared memory the CTA no longer owns.
// (Copying the owner's own rank's first tiles before the arrival barrier, to
// overlap the pipeline fill with the flag round trip, made the barrier
// itself 1.5-2.3 us slower on GB300: the burst of reads delayed the flags.)
// No multicast and no bulk reduction (its order of additions is not fixed).
// Streaming copies carry an L2 evict-first hint: every byte is touched once.
//
// Synchronisation between simulated ranks (the pages' counters reaching N,
// page 1 section "Four barrier-free mechanisms", part 4, kept as flags):
//   * arrival (top barrier): CTA (q, k) stores its epoch into arrive[q][k];
//     owners read rank q's input and write rank q's output only once every
//     rank has arrived at this call;
//   * completion: after its bulk stores have completed, owner j stores the
//     epoch into cmpl[p][j][k] for every rank p, and CTA (p, k) waits for
//     all owners before it reports its call finished.
// No receive buffers, so nothing to double-buffer and no bottom barrier.
#include "sfar_prims.cuh"

#define TMA_OUT_BUFS 3

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(phase)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t pol)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src, uint32_t bytes, uint64_t pol)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst), "r"(src),
                 "r"(bytes), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// Wait for phase `parity`, bounded by time only (not by the status word: it
// is used after a failure, to let copies already issued land).
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((it & 127u) == 0 && globaltimer() - t0 > limit_ns)
            return false;
    }
}
// Poll a flag of another rank until it reaches epoch e, with acquire loads
// (the CTA barrier after the exchange passes the acquisition on); false if
// the bounded wait gave up.
__device__ __forceinline__ bool poll_acquire_ge(const uint32_t *f, uint32_t e, const SfarCtl *ctl, bool downstream)
{
    SfarWaiter w(downstream);
    while (!epoch_ge(ld_acquire_u32(f), e))
        if (w.tick(ctl))
            return false;
    return true;
}
// Bounded wait for phase `parity` of an mbarrier; false if it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const SfarCtl *ctl)
{
    SfarWaiter w;
    while (!mbar_try_wait(bar, parity))
        if (w.tick(ctl))
            return false;
    return true;
}

#define TMA_CONSUMER_WARPS 8
#define TMA_PRODUCER_WARP 8
#define TMA_STORE_WARP 9

template <int DT, bool TEST>
__global__ void __launch_bounds__(SFAR_TMA_THREADS, 1) k_tma(const __grid_constant__ SfarArgs a)
{
    constexpr int ES = DT == 0 ? 2 : 4;
    constexpr int NB = TMA_OUT_BUFS;
    // Early ticket (see sfar_entry): the epoch atomic overlaps the wait for the
    // predecessor.  A successor cannot start on this kernel's SMs anyway (its
    // shared memory fills them), so launching it earlier costs nothing here.
    const SfarEntry ent = sfar_entry<true>(a);
    const int R = a.R, K = a.K;
    const int r = blockIdx.x / K, k = blockIdx.x - r * K;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    SfarCall c;
    if (!sfar_prologue<TEST>(a, r, k, c, ent))
        return;
    const uint32_t e = c.e;
    uint32_t *arrive = a.fa;      // [R][KMAX]
    uint32_t *cmpl = a.fb;        // [receiver][owner][KMAX]
    __shared__ int s_ok;

    // arrival: this rank's input is ready and its output free for this call
    if (tid < 32) {
        if (tid == 0 && !c.drop)
            st_release_u32(arrive + sfar_pull_flag(r, k), e);
        int ok = 1;
        for (int i = lane; i < R - 1 && ok; i += 32) {
            const int q = peer_of(r, i);
            if (!poll_acquire_ge(arrive + sfar_pull_flag(q, k), e, a.ctl, false)) {
                sfar_record_fault(a.ctl, r, k, q, e, SFAR_WAIT_ARRIVE);
                ok = 0;
            }
        }
        ok = __all_sync(SFAR_FULL, ok);
        if (tid == 0)
            s_ok = ok;
    }
    __syncthreads();
    bool ok = s_ok != 0;
    sfar_mid_delay<TEST>(c);
    sfar_stamp(c, TP_SENT);

    // this CTA's byte range [b0, b1) of chunk r
    const unsigned long long nbytes = a.n * ES;
    const unsigned long long cb0 = (unsigned long long)r * a.chunk * ES;
    unsigned long long b0 = cb0 + (unsigned long long)k * a.sub * ES;
    unsigned long long b1 = b0 + a.sub * ES;
    const unsigned long long cb1 = cb0 + a.chunk * ES;
    if (b1 > cb1) b1 = cb1;
    if (b1 > nbytes) b1 = nbytes;
    if (b0 > b1) b0 = b1;
    const unsigned long long len16 = (b1 - b0) & ~15ull;
    const uint32_t TB = (uint32_t)a.tile_bytes;
    const int NS = a.stages;
    const unsigned long long ntiles = (len16 + TB - 1) / TB;

    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *stage0 = smem;                                           // [NS][R][TB]
    uint8_t *obuf = smem + (size_t)NS * R * TB;                       // [NB][TB]
    uint64_t *full = reinterpret_cast<uint64_t *>(obuf + (size_t)NB * TB);   // [NS]
    uint64_t *empty = full + NS;                                      // [NS]
    uint64_t *ofull = empty + NS;                                     // [NB]
    uint64_t *ofree = ofull + NB;                                     // [NB]
    __shared__ int s_fail;

    if (ok && ntiles > 0) {
        if (tid == 0) {
            for (int s = 0; s < NS; ++s) {
                mbar_init(smem_u32(full + s), 1);
                mbar_init(smem_u32(empty + s), TMA_CONSUMER_WARPS);
            }
            for (int b = 0; b < NB; ++b) {
                mbar_init(smem_u32(ofull + b), TMA_CONSUMER_WARPS);
                mbar_init(smem_u32(ofree + b), 1);
            }
            s_fail = 0;
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            fence_proxy_async_smem();
        }
        __syncthreads();
        const auto tile_len = [&](unsigned long long t) {
            const unsigned long long off = t * TB;
            return (uint32_t)((len16 - off) < TB ? (len16 - off) : TB);
        };
        unsigned long long issued = 0;  // producer: tiles whose copies went out
        if (warp == TMA_PRODUCER_WARP) {
            const uint64_t pol = policy_evict_first();
            unsigned long long t = 0;
            for (; t < ntiles; ++t) {
                const int s = (int)(t % NS);
                int wok = 1;
                if (t >= (unsigned long long)NS)
                    wok = mbar_wait(smem_u32(empty + s), (uint32_t)(((t / NS) - 1) & 1ull), a.ctl);
                if (!__all_sync(SFAR_FULL, wok)) {
                    if (lane == 0) {
                        sfar_record_fault(a.ctl, r, k, -1, e, SFAR_WAIT_COPY);
                        s_fail = 1;
                    }
                    break;
                }
                const uint32_t tb = tile_len(t), bar = smem_u32(full + s);
                if (lane == 0)
                    mbar_expect_tx(bar, tb * (uint32_t)R);
                __syncwarp();
                for (int q = lane; q < R; q += 32)
                    bulk_g2s(smem_u32(stage0 + ((size_t)s * R + q) * TB), (const uint8_t *)a.in[q] + b0 + t * TB, tb,
                             bar, pol);
            }
            issued = t;
        } else if (warp == TMA_STORE_WARP) {
            const uint64_t pol = policy_evict_first();
            for (unsigned long long t = 0; t < ntiles; ++t) {
                const int b = (int)(t % NB);
                const int wok = mbar_wait(smem_u32(ofull + b), (uint32_t)((t / NB) & 1ull), a.ctl);
                if (!__all_sync(SFAR_FULL, wok)) {
                    if (lane == 0) {
                        sfar_record_fault(a.ctl, r, k, -1, e, SFAR_WAIT_COPY);
                        s_fail = 1;
                    }
                    break;
                }
                const uint32_t tb = tile_len(t);
                for (int p = lane; p < R; p += 32)
                    bulk_s2g((uint8_t *)a.out[p] + b0 + t * TB, smem_u32(obuf + (size_t)b * TB), tb, pol);
                bulk_commit();
                // the copies of tile t - 1 have read their buffer: free it
                bulk_wait_read1();
                __syncwarp();
                if (t >= 1 && lane == 0)
                    mbar_arrive(smem_u32(ofree + (int)((t - 1) % NB)));
            }
            bulk_wait0();               // stores complete before completion is signalled
            fence_proxy_async_global();
        } else {
            const int ct = tid;         // consumer threads 0 .. 32 * TMA_CONSUMER_WARPS - 1
            for (unsigned long long t = 0; t < ntiles; ++t) {
                const int s = (int)(t % NS), b = (int)(t % NB);
                int wok = mbar_wait(smem_u32(full + s), (uint32_t)((t / NS) & 1ull), a.ctl);
                if (wok && t >= (unsigned long long)NB)
                    wok = mbar_wait(smem_u32(ofree + b), (uint32_t)(((t / NB) - 1) & 1ull), a.ctl);
                if (!__all_sync(SFAR_FULL, wok)) {
                    if (lane == 0) {
                        sfar_record_fault(a.ctl, r, k, -1, e, SFAR_WAIT_COPY);
                        s_fail = 1;
                    }
                    break;
                }
                const uint32_t tb = tile_len(t);
                const uint8_t *st = stage0 + (size_t)s * R * TB;
                uint8_t *ob = obuf + (size_t)b * TB;
                for (uint32_t u = ct * 16u; u < tb; u += TMA_CONSUMER_WARPS * 32 * 16u) {
                    SfarAcc<DT> acc;
                    acc.set(*reinterpret_cast<const uint4 *>(st + u));
                    for (int q = 1; q < R; ++q)
                        acc.add(*reinterpret_cast<const uint4 *>(st + (size_t)q * TB + u));
                    *reinterpret_cast<uint4 *>(ob + u) = acc.get();
                }
                fence_proxy_async_smem();   // our writes to the buffer, before the bulk stores read it
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(smem_u32(empty + s));
                    mbar_arrive(smem_u32(ofull + b));
                }
            }
        }
        __syncthreads();
        ok = ok && s_fail == 0;
        if (!ok && warp == TMA_PRODUCER_WARP && lane == 0) {
            // a wait gave up somewhere in the CTA: let the copies already
            // issued land before the shared memory is released (the last tile
            // issued into a slot completes after every earlier one there)
            const unsigned long long limit_ns = ld_relaxed_u64(&a.ctl->timeout_ns);
            for (int s = 0; s < NS && (unsigned long long)s < issued; ++s) {
                const unsigned long long last = issued - 1 - ((issued - 1 - s) % NS);
                mbar_wait_for(smem_u32(full + s), (uint32_t)((last / NS) & 1ull), limit_ns);
            }
        }
    }
    // a ragged end shorter than 16 bytes: element by element
    if (ok && tid == 0 && b1 == nbytes && (b1 - b0) > len16) {
        for (unsigned long long bb = b0 + len16; bb < b1; bb += ES) {
            float acc = 0.f;
            for (int q = 0; q < R; ++q) {
                float x;
                if (ES == 2)
                    x = __uint_as_float((uint32_t)(*(const uint16_t *)((const uint8_t *)a.in[q] + bb)) << 16);
                else
                    x = *(const float *)((const uint8_t *)a.in[q] + bb);
                acc = q == 0 ? x : __fadd_rn(acc, x);
            }
            for (int p = 0; p < R; ++p) {
                if (ES == 2) {
                    __nv_bfloat16 h = __float2bfloat16_rn(acc);
                    *(uint16_t *)((uint8_t *)a.out[p] + bb) = *reinterpret_cast<uint16_t *>(&h);
                } else {
                    *(float *)((uint8_t *)a.out[p] + bb) = acc;
                }
            }
        }
    }
    __syncthreads();
    sfar_stamp(c, TP_INPUT);        // this path: the CTA's tiles are folded and stored
    // completion: tell every rank this owner's part of its output is written
    // (release stores after the CTA barrier that follows the store warp's
    // bulk-store wait and proxy fence; acquire polls, passed on to the CTA by
    // the epilogue's barrier)
    if (tid < 32) {
        if (ok && !c.drop)
            for (int p = lane; p < R; p += 32)
                if (p != r)
                    st_release_u32(cmpl + sfar_pull_flag((size_t)p * R + r, k), e);
        int wok = ok ? 1 : 0;
        for (int i = lane; i < R - 1 && wok; i += 32) {
            const int q = peer_of(r, i);
            if (!poll_acquire_ge(cmpl + sfar_pull_flag((size_t)r * R + q, k), e, a.ctl, true)) {
                sfar_record_fault(a.ctl, r, k, q, e, SFAR_WAIT_COMPLETE);
                wok = 0;
            }
        }
        __syncwarp();
    }
    sfar_stamp(c, TP_RECEIVED);
    sfar_epilogue(a, r, k, e);
    sfar_stamp(c, TP_EXIT);
}

const void *sfar_kernel_tma(int dt, int test)
{
    if (dt == 0)
        return test ? (const void *)k_tma<0, true> : (const void *)k_tma<0, false>;
    return test ? (const void *)k_tma<1, true> : (const void *)k_tma<1, false>;
}
