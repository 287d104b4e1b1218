// sfar_prims.cuh -- device primitives of libsfar (sm_103a).
//
// These are the building blocks the pages name for their LLBuffer object
// ("Every Microsecond Counts" (page 1), section "Unified primitives and API
// design": send to a peer's slot, recv by polling a slot until its data is
// valid, recvReduce summing several peers in registers, reset of the slots,
// and an epoch advanced once per collective).  Here they are inline
// functions over plain global-memory slots:
//   * memory-ordered accesses written as inline PTX (ld/st .relaxed.gpu,
//     .release.gpu, .acquire.gpu, fence.acq_rel.gpu);
//   * bounded polling: every wait reads %globaltimer now and then and gives
//     up after the handle's limit, recording where in the status block, so a
//     lost message never hangs the GPU;
//   * the per-call prologue/epilogue: epoch ticket, overlap-mode hand-off
//     between consecutive calls of the same (rank, CTA), test knobs;
//   * the fixed-order reduction: binary32 accumulator, left fold in rank
//     order, one round-to-nearest-even to the element type;
//   * the LL packet and LL128 line layouts.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "sfar.h"
#include "sfar_internal.h"

#define SFAR_FULL 0xffffffffu

// ---------------------------------------------------------------- PTX access
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ int ld_relaxed_s32(const int *p)
{
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p)
{
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u32(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_release_u32(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu()
{
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ uint4 ld_relaxed_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_v4(void *p, uint4 v)
{
    asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
// Two 8-byte words in one instruction; each word is single-copy atomic.
__device__ __forceinline__ void ld_relaxed_v2u64(const void *p, unsigned long long &a,
                                                 unsigned long long &b)
{
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0,%1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_relaxed_v2u64(void *p, unsigned long long a, unsigned long long b)
{
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1,%2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
// Plain (weak) accesses for data that a flag orders.
__device__ __forceinline__ void st_v4(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_u32(void *p, uint32_t v)
{
    asm volatile("st.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_v2u32(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}
// Read-only input of the calling rank (not written while the kernel runs).
__device__ __forceinline__ uint4 ld_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Programmatic dependent launch: lets the next kernel on the stream start.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Waits until every prerequisite grid has completed and its memory is visible
// (a no-op when the kernel was launched without a programmatic dependency).
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Brings a line into L2 (and its translation into the TLBs) without
// returning data.  Safe before griddepcontrol.wait: L2 is the point of
// coherence, so a later write by the previous kernel still updates the line.
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// Trace stamps of one CTA (thread 0): kernel entry, and the moment the
// programmatic-launch wait returned.  Recorded only when tracing is armed.
struct SfarEntry {
    unsigned long long t_entry, t_start;
    unsigned long long ticket;    // serial mode, thread 0: the rank counter before this CTA's add
    bool have_ticket;
};

__device__ __forceinline__ unsigned long long sfar_take_ticket(const SfarArgs &a, int r, int k)
{
    // Every CTA of rank r adds to the rank's call counter: CTA 0 adds
    // SFAR_KMAX - K + 1, the others 1, so each call adds exactly SFAR_KMAX and
    // every CTA of call c (counted from 0) receives a value in
    // [c * SFAR_KMAX, (c + 1) * SFAR_KMAX) whatever the order of the atomics:
    // all CTAs agree on the epoch c + 1, and the epoch is the same for every
    // launch geometry.
    const unsigned long long add = k == 0 ? (unsigned long long)(SFAR_KMAX - a.K + 1) : 1ull;
    return atomicAdd(a.epoch + r, add);
}

// First statement of every AllReduce kernel.  In serial mode the kernel is
// launched as a programmatic dependent of the previous kernel on the stream
// and waits here for its predecessor to complete, so it sees exactly what
// plain stream order would show it; the prologue then lets its own successor
// be scheduled once every CTA holds its ticket, so the successor's launch
// overlaps this kernel's work while at most one launched kernel waits.
// With EARLY, thread 0 takes its ticket before the wait: the predecessor
// lets this kernel launch only after every one of its CTAs has received its
// own ticket, and nothing else touches the counters (sfar_reset clears them
// with plain stream order), so the atomic's round trip overlaps the wait.
// Measured on GB300 (R = 8, 16 KB): DB 4.48 -> 4.20 us, BASELINE 6.04 ->
// 5.85, sentinel 3.21 -> 3.14, LL128 4.85 -> 4.83, but LL 3.20 -> 3.39 (its
// successor then launches earlier, into its receive), so each kernel chooses.
// In overlap mode the kernel does not wait (the prologue hands off inside
// one rank instead) and the prologue takes the ticket.
template <bool EARLY = false>
__device__ __forceinline__ SfarEntry sfar_entry(const SfarArgs &a)
{
    SfarEntry t{0, 0, 0, false};
    const bool tr = a.trace != nullptr && threadIdx.x == 0;
    if (tr)
        t.t_entry = globaltimer();
    if (!a.overlap) {
        if (EARLY && threadIdx.x == 0) {
            const int r = blockIdx.x / a.K;
            t.ticket = sfar_take_ticket(a, r, blockIdx.x - r * a.K);
            t.have_ticket = true;
        }
        pdl_wait();
    }
    if (tr)
        t.t_start = globaltimer();
    return t;
}

// ------------------------------------------------------------ bounded waits
// Records status `code` (the first failure wins) with where it happened.
__device__ __forceinline__ void sfar_record_code(SfarCtl *ctl, int code, int rank, int cta, int peer, uint32_t e,
                                                 int where)
{
    if (atomicCAS(&ctl->status, 0, code) == 0) {
        volatile SfarCtl *c = ctl;
        c->f_rank = rank;
        c->f_cta = cta;
        c->f_peer = peer;
        c->f_epoch = e;
        c->f_where = where;
    }
}

// A bounded wait gave up: SFAR_ERR_TIMEOUT.
__device__ __forceinline__ void sfar_record_fault(SfarCtl *ctl, int rank, int cta, int peer, uint32_t e,
                                                  int where)
{
    sfar_record_code(ctl, SFAR_ERR_TIMEOUT, rank, cta, peer, e, where);
}

// One waiter per poll loop.  tick() is cheap on the fast path (a counter);
// every 128 iterations it reads %globaltimer, gives up after the limit, and
// also gives up at once if another CTA has already recorded a failure.
// Waits that can only fail because an earlier wait failed (completion,
// all-gather, bottom barrier, the overlap hand-off) are "downstream" and get
// twice the limit, so the first failure recorded is the root cause.
struct SfarWaiter {
    unsigned long long t0;
    uint32_t it;
    int shift;
    __device__ __forceinline__ SfarWaiter(bool downstream = false) : t0(0), it(0), shift(downstream ? 1 : 0) {}
    __device__ __forceinline__ bool tick(const SfarCtl *ctl)
    {
        if ((++it & 127u) != 0)
            return false;
        const unsigned long long now = globaltimer();
        if (t0 == 0) {
            t0 = now;
            return false;
        }
        if (ld_relaxed_s32(&ctl->status) != 0)
            return true;
        return now - t0 > (ld_relaxed_u64(&ctl->timeout_ns) << shift);
    }
};

// epoch compare that survives wrap-around: a >= b
__device__ __forceinline__ bool epoch_ge(uint32_t a, uint32_t b) { return (int32_t)(a - b) >= 0; }

// Poll a u32 flag until it reaches epoch e (relaxed loads; the caller fences).
__device__ __forceinline__ bool poll_flag_ge(const uint32_t *f, uint32_t e, const SfarCtl *ctl,
                                             bool downstream = false)
{
    SfarWaiter w(downstream);
    while (!epoch_ge(ld_relaxed_u32(f), e))
        if (w.tick(ctl))
            return false;
    return true;
}

// ------------------------------------------------------- prologue / epilogue
struct SfarCall {
    uint32_t e;     // this call's epoch (1, 2, ...) for (rank, CTA)
    int par;        // receive-buffer parity
    bool drop;      // test knob: this rank sends nothing
    uint32_t mid_delay_ns;       // test knob: straggler delay between sends and receives
    unsigned long long *trace;   // this CTA's trace entry for this call (thread 0 only), or NULL
};

// Trace points (thread 0's view); slot TP_EPOCH holds the epoch itself.
enum {
    TP_ENTRY = 0,      // kernel entry
    TP_START = 1,      // programmatic-launch wait returned (serial mode)
    TP_TICKET = 2,     // epoch known (overlap mode: after the hand-off)
    TP_INPUT = 3,      // first input vector arrived
    TP_SENT = 4,       // sends issued (DB / baseline: top barrier passed)
    TP_RECEIVED = 5,   // receive and reduction done
    TP_EXIT = 6,       // last statement
    TP_EPOCH = 7
};

__device__ __forceinline__ void sfar_stamp(const SfarCall &c, int point)
{
    if (c.trace)
        c.trace[point] = globaltimer();
}

// Stamp once the value `dep` has arrived (the asm consumes it first).
__device__ __forceinline__ void sfar_stamp_after(const SfarCall &c, int point, uint32_t dep)
{
    if (c.trace) {
        uint32_t sink;
        asm volatile("mov.b32 %0, %1;" : "=r"(sink) : "r"(dep));
        c.trace[point] = globaltimer() + (sink & 0u);
    }
}

__device__ __forceinline__ void spin_ns(unsigned long long d)
{
    const unsigned long long t0 = globaltimer();
    while (globaltimer() - t0 < d) {
    }
}

// Every thread of the CTA calls this.  Returns false if the CTA must exit at
// once (the handle already holds a failure, or a wait gave up here).
template <bool TEST>
__device__ __forceinline__ bool sfar_prologue(const SfarArgs &a, int r, int k, SfarCall &c, const SfarEntry &t)
{
    __shared__ uint32_t s_e;
    __shared__ int s_flags;
    c.trace = nullptr;
    if (threadIdx.x == 0) {
        // Ticket (sfar_take_ticket).  Calls never interleave their tickets
        // (stream order, or the launch of the next call after every CTA of
        // this one holds its ticket).  In serial mode it was taken before the
        // programmatic-launch wait; in overlap mode its latency overlaps the
        // input load the caller issued just before.
        const unsigned long long tk = t.have_ticket ? t.ticket : sfar_take_ticket(a, r, k);
        const uint32_t e = (uint32_t)(tk / SFAR_KMAX) + 1u;
        int flags = ld_relaxed_s32(&a.ctl->status) != 0 ? 1 : 0;
        if (TEST) {
            const volatile SfarCtl *ctl = a.ctl;
            if (ctl->drop_rank == r)
                flags |= 2;
            if (ctl->single_buffer)
                flags |= 4;
        }
        s_e = e;
        s_flags = flags;
        if (a.trace) {
            c.trace = a.trace + ((size_t)(e % a.trace_calls) * gridDim.x + blockIdx.x) * SFAR_TRACE_POINTS;
            c.trace[TP_ENTRY] = t.t_entry;
            c.trace[TP_START] = t.t_start;
            c.trace[TP_EPOCH] = e;
        }
    }
    __syncthreads();
    c.e = s_e;
    const int flags = s_flags;
    // The successor may take its tickets only after all of ours are taken
    // (a successor in overlap mode does not wait for this kernel to end).
    // A solo grid (one that fills the GPU) lets it launch only at its end.
    if ((!a.overlap || (flags & 1)) && !a.solo)
        pdl_launch_dependents();
    if (flags & 1)
        return false;
    c.drop = (flags & 2) != 0;
    c.par = (flags & 4) ? 0 : (int)(c.e & 1u);
    c.mid_delay_ns = 0;
    if (a.overlap || TEST) {
        __shared__ int s_ok;
        __shared__ uint32_t s_mid;
        if (threadIdx.x == 0) {
            int ok = 1;
            if (a.overlap) {
                // wait for CTA (r, k) of the previous call: a wait inside one rank
                SfarWaiter w(true);
                const uint32_t *d = a.done + r * SFAR_KMAX + k;
                while (!epoch_ge(ld_acquire_u32(d), c.e - 1u)) {
                    if (w.tick(a.ctl)) {
                        sfar_record_fault(a.ctl, r, k, -1, c.e, SFAR_WAIT_DONE);
                        ok = 0;
                        break;
                    }
                }
            }
            uint32_t mid = 0;
            if (TEST && ok) {
                const volatile SfarCtl *ctl = a.ctl;
                const uint32_t len = ctl->strag_len;
                if (len) {
                    const uint32_t idx = c.e - ctl->strag_base - 1u;
                    const int who = ctl->strag_rank < 0 ? (int)(idx % (uint32_t)a.R) : ctl->strag_rank;
                    if (who == r && idx < 0x40000000u) {
                        const uint32_t d = ctl->strag_delays[idx % len];
                        if (ctl->strag_phase == 0)
                            spin_ns(d);
                        else
                            mid = d;
                    }
                }
            }
            s_ok = ok;
            s_mid = mid;
        }
        __syncthreads();
        // Overlap mode: the next call's kernel may start once every CTA of
        // this one holds its ticket and has seen its predecessor (r, k) done,
        // which keeps at most two calls ahead of the oldest running one.
        if (a.overlap)
            pdl_launch_dependents();
        if (!s_ok)
            return false;
        c.mid_delay_ns = s_mid;
    }
    sfar_stamp(c, TP_TICKET);
    return true;
}

// Test variants: a straggler of phase 1 waits here, after its sends and
// before it reads anything it received.
template <bool TEST>
__device__ __forceinline__ void sfar_mid_delay(const SfarCall &c)
{
    if (TEST && c.mid_delay_ns) {
        if (threadIdx.x == 0)
            spin_ns(c.mid_delay_ns);
        __syncthreads();
    }
}

// Marks (rank, CTA) done with epoch e.  In overlap mode the next call's CTA
// (r, k) acquires it, so it is a release after a CTA barrier; in serial mode
// the kernel boundary orders everything and a relaxed store suffices.
__device__ __forceinline__ void sfar_epilogue(const SfarArgs &a, int r, int k, uint32_t e)
{
    if (a.overlap) {
        __syncthreads();
        if (threadIdx.x == 0)
            st_release_u32(a.done + r * SFAR_KMAX + k, e);
    } else if (threadIdx.x == 0) {
        st_relaxed_u32(a.done + r * SFAR_KMAX + k, e);
    }
}

// ------------------------------------------------ element vectors (16 bytes)
// Load 16 bytes of a rank's input; bytes past nbytes read as zero, element by
// element, so a ragged tail never reads past the caller's buffer.
template <int ES>
__device__ __forceinline__ uint4 load_vec(const void *base, unsigned long long v, unsigned long long nbytes)
{
    const unsigned long long off = v * 16ull;
    if (off + 16ull <= nbytes)
        return ld_nc_v4((const char *)base + off);
    uint32_t w0 = 0, w1 = 0, w2 = 0, w3 = 0;
    if (off < nbytes) {
        const char *p = (const char *)base + off;
        const int rem = (int)(nbytes - off);
        if (ES == 4) {
            const uint32_t *q = (const uint32_t *)p;
            if (rem > 0) w0 = q[0];
            if (rem > 4) w1 = q[1];
            if (rem > 8) w2 = q[2];
        } else {
            const uint16_t *q = (const uint16_t *)p;
            if (rem > 0) w0 = q[0];
            if (rem > 2) w0 |= (uint32_t)q[1] << 16;
            if (rem > 4) w1 = q[2];
            if (rem > 6) w1 |= (uint32_t)q[3] << 16;
            if (rem > 8) w2 = q[4];
            if (rem > 10) w2 |= (uint32_t)q[5] << 16;
            if (rem > 12) w3 = q[6];
        }
    }
    return make_uint4(w0, w1, w2, w3);
}

template <int ES>
__device__ __forceinline__ void store_vec(void *base, unsigned long long v, unsigned long long nbytes, uint4 x)
{
    const unsigned long long off = v * 16ull;
    if (off + 16ull <= nbytes) {
        st_v4((char *)base + off, x);
        return;
    }
    if (off >= nbytes)
        return;
    char *p = (char *)base + off;
    const int rem = (int)(nbytes - off);
    if (ES == 4) {
        uint32_t *q = (uint32_t *)p;
        if (rem > 0) q[0] = x.x;
        if (rem > 4) q[1] = x.y;
        if (rem > 8) q[2] = x.z;
    } else {
        uint16_t *q = (uint16_t *)p;
        if (rem > 0) q[0] = (uint16_t)x.x;
        if (rem > 2) q[1] = (uint16_t)(x.x >> 16);
        if (rem > 4) q[2] = (uint16_t)x.y;
        if (rem > 6) q[3] = (uint16_t)(x.y >> 16);
        if (rem > 8) q[4] = (uint16_t)x.z;
        if (rem > 10) q[5] = (uint16_t)(x.z >> 16);
        if (rem > 12) q[6] = (uint16_t)x.w;
    }
}

// ---------------------------------------------------- fixed-order reduction
// Accumulator of one 16-byte vector: 8 bf16 or 4 fp32 elements held as
// binary32.  set() takes rank 0's value, add() each later rank in order;
// every add rounds to nearest even (__fadd_rn: never contracted, never
// flushed); get() rounds once to the element type.
template <int DT> struct SfarAcc;

template <> struct SfarAcc<0> {
    float v[8];
    __device__ __forceinline__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
    __device__ __forceinline__ static float hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
    __device__ __forceinline__ void set(uint4 x)
    {
        v[0] = lo(x.x); v[1] = hi(x.x); v[2] = lo(x.y); v[3] = hi(x.y);
        v[4] = lo(x.z); v[5] = hi(x.z); v[6] = lo(x.w); v[7] = hi(x.w);
    }
    __device__ __forceinline__ void add(uint4 x)
    {
        v[0] = __fadd_rn(v[0], lo(x.x)); v[1] = __fadd_rn(v[1], hi(x.x));
        v[2] = __fadd_rn(v[2], lo(x.y)); v[3] = __fadd_rn(v[3], hi(x.y));
        v[4] = __fadd_rn(v[4], lo(x.z)); v[5] = __fadd_rn(v[5], hi(x.z));
        v[6] = __fadd_rn(v[6], lo(x.w)); v[7] = __fadd_rn(v[7], hi(x.w));
    }
    __device__ __forceinline__ static uint32_t pack(float a, float b)
    {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);   // .x (low half) = a
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ uint4 get() const
    {
        return make_uint4(pack(v[0], v[1]), pack(v[2], v[3]), pack(v[4], v[5]), pack(v[6], v[7]));
    }
};

template <> struct SfarAcc<1> {
    float v[4];
    __device__ __forceinline__ void set(uint4 x)
    {
        v[0] = __uint_as_float(x.x); v[1] = __uint_as_float(x.y);
        v[2] = __uint_as_float(x.z); v[3] = __uint_as_float(x.w);
    }
    __device__ __forceinline__ void add(uint4 x)
    {
        v[0] = __fadd_rn(v[0], __uint_as_float(x.x)); v[1] = __fadd_rn(v[1], __uint_as_float(x.y));
        v[2] = __fadd_rn(v[2], __uint_as_float(x.z)); v[3] = __fadd_rn(v[3], __uint_as_float(x.w));
    }
    __device__ __forceinline__ uint4 get() const
    {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                          __float_as_uint(v[3]));
    }
};

// Rank index of the i-th peer of rank r (peers in rank order, r skipped).
__device__ __forceinline__ int peer_of(int r, int i) { return i < r ? i : i + 1; }

// --------------------------------------------------------------- LL packets
// One 16-byte input vector (words w0..w3) travels as two 16-byte LL lines,
// each two 8-byte words {data, flag}: single-copy atomic per 8-byte word, so
// a reader that sees flag == e in a word also sees that word's data.
__device__ __forceinline__ bool ll_ready(unsigned long long a, unsigned long long b, unsigned long long c,
                                         unsigned long long d, uint32_t e)
{
    return (uint32_t)(a >> 32) == e && (uint32_t)(b >> 32) == e && (uint32_t)(c >> 32) == e &&
           (uint32_t)(d >> 32) == e;
}

// ------------------------------------------------------------- LL128 lines
// A warp moves 4 lines of 128 bytes at once: line g (g = lane / 8) is held by
// lanes 8g..8g+7, 16 bytes each; word 0 of each line is its flag, the other
// 31 words carry 31 consecutive payload words.  The 124 payload words of the
// 4 lines are the 31 consecutive 16-byte input vectors held by lanes 0..30.
__device__ __forceinline__ uint4 shfl4(uint4 x, int src)
{
    x.x = __shfl_sync(SFAR_FULL, x.x, src);
    x.y = __shfl_sync(SFAR_FULL, x.y, src);
    x.z = __shfl_sync(SFAR_FULL, x.z, src);
    x.w = __shfl_sync(SFAR_FULL, x.w, src);
    return x;
}
// word i (0..7) of the 8-word sequence A, B
__device__ __forceinline__ uint32_t pick8(const uint4 &A, const uint4 &B, int i)
{
    const uint32_t a01 = (i & 1) ? A.y : A.x, a23 = (i & 1) ? A.w : A.z;
    const uint32_t b01 = (i & 1) ? B.y : B.x, b23 = (i & 1) ? B.w : B.z;
    const uint32_t a = (i & 2) ? a23 : a01, b = (i & 2) ? b23 : b01;
    return (i & 4) ? b : a;
}
// vector layout (lane l < 31 holds payload words 4l..4l+3) -> line layout
// (this lane's 16 bytes of the 4 lines; word 0 of a line slot is left for the flag)
__device__ __forceinline__ uint4 ll128_pack(uint4 x, int lane)
{
    const int g = lane >> 3, m = lane & 7;
    const int s = 31 * g + 4 * m - 1;           // payload word under this slot's word 0
    const int a = (s + 4) / 4 - 1;              // floor(s / 4), s >= -1
    const int c = s - 4 * a;
    const uint4 A = shfl4(x, a & 31), B = shfl4(x, (a + 1) & 31);
    return make_uint4(pick8(A, B, c), pick8(A, B, c + 1), pick8(A, B, c + 2), pick8(A, B, c + 3));
}
// line layout -> vector layout (valid on lanes 0..30)
__device__ __forceinline__ uint4 ll128_unpack(uint4 y, int lane)
{
    const int w0 = 4 * lane;
    const int x0 = w0 + w0 / 31 + 1;           // line-word index of payload word w0
    const int a = x0 >> 2;
    const uint4 A = shfl4(y, a & 31), B = shfl4(y, (a + 1) & 31);
    uint32_t o[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const int w = w0 + t;
        o[t] = pick8(A, B, w + w / 31 + 1 - 4 * a);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}
// Store this lane's 16 bytes of a line, leaving the flag word alone.
__device__ __forceinline__ void ll128_store_data(uint8_t *line, int m, uint4 y)
{
    if (m != 0) {
        st_v4(line + 16 * m, y);
    } else {
        st_u32(line + 4, y.y);
        st_v2u32(line + 8, y.z, y.w);
    }
}
