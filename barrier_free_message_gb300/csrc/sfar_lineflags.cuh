// sfar_lineflags.cuh -- the wait for the line flags of the LL128 kernels
// (the one-shot k_ll128 and the two-shot k_twoshot).
//
// "Every Microsecond Counts" (page 1), section "Four barrier-free
// mechanisms", part 4: a reader waits until a 128-byte line's flag holds the
// call's epoch, then reads the line.  Lane (g, m) of a warp waits for line g
// of peers m and m + 8 (those below R - 1).
#pragma once
#include "sfar_prims.cuh"

// base: the reader's region of this call's parity, one slot of `slot` bytes
// per sender; loff: the line's offset in a slot.  Returns false, after
// recording the fault at `where`, if the bounded wait gave up.  With at most
// 8 peers a lane has one flag and polls it with acquire loads.  With more, a
// lane reads both of its flags in every round with relaxed loads (two acquire
// loads would wait for each other) and closes the acquisition with one
// acquire fence (fence.acquire: unlike fence.acq_rel it does not wait for the
// lane's earlier stores, the previous line group's sends).  Either way the
// caller passes each lane's acquisition on to the warp with __syncwarp before
// the warp reads the lines.
template <int RB>
__device__ __forceinline__ bool wait_line_flags(const uint8_t *base, size_t slot, size_t loff, int r, int R, int m,
                                                uint32_t e, SfarCtl *ctl, int k, int where, bool downstream)
{
    if (RB <= 8) {
        for (int i = m; i < R - 1; i += 8) {
            const int q = peer_of(r, i);
            const uint32_t *f = (const uint32_t *)(base + (size_t)q * slot + loff);
            SfarWaiter w(downstream);
            while (ld_acquire_u32(f) != e)
                if (w.tick(ctl)) {
                    sfar_record_fault(ctl, r, k, q, e, where);
                    return false;
                }
        }
        return true;
    }
    const int q0 = m < R - 1 ? peer_of(r, m) : -1, q1 = m + 8 < R - 1 ? peer_of(r, m + 8) : -1;
    const uint32_t *f0 = (const uint32_t *)(base + (size_t)(q0 < 0 ? 0 : q0) * slot + loff);
    const uint32_t *f1 = (const uint32_t *)(base + (size_t)(q1 < 0 ? 0 : q1) * slot + loff);
    bool d0 = q0 < 0, d1 = q1 < 0;
    SfarWaiter w(downstream);
    while (!(d0 && d1)) {
        const uint32_t v0 = d0 ? e : ld_relaxed_u32(f0);
        const uint32_t v1 = d1 ? e : ld_relaxed_u32(f1);
        d0 = v0 == e;
        d1 = v1 == e;
        if (!(d0 && d1) && w.tick(ctl)) {
            sfar_record_fault(ctl, r, k, d0 ? q1 : q0, e, where);
            return false;
        }
    }
    asm volatile("fence.acquire.gpu;" ::: "memory");
    return true;
}
