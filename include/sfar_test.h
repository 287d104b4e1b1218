/*
 * sfar_test.h -- test and measurement hooks of libsfar.
 *
 * Nothing here is needed to use the AllReduce.  The hooks let tests and the
 * benchmark delay a simulated rank, drop a rank's sends, shorten the device
 * wait limit, switch the launch mode and time the latency floor.  Each knob
 * is a field of the handle's device status block, written by a one-thread
 * kernel on the given stream, so it takes effect for calls enqueued after it
 * on that stream.  Calls made while a knob is armed run a kernel variant that
 * reads the knobs; otherwise the kernels never read them.
 */
#ifndef SFAR_TEST_H
#define SFAR_TEST_H

#include "sfar.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Straggler injection.  The straggler of a workload is the last-arriving
 * rank, and it sets the latency ("SiFAR" (page 3), sections "Technique 3"
 * and "Limitations"; the tail-latency discussion of the small-message page).
 * From the next call on, call i (counted per CTA from the arming point)
 * delays every CTA of rank (rank < 0 ? i mod R : rank) by delays_ns[i mod len]
 * nanoseconds (a spin on %globaltimer).  phase 0: the delay comes before the
 * rank sends anything (a late arrival).  phase 1: it comes after the rank's
 * sends and before it reads what it received (a slow reader, the case in
 * which a peer that has moved on could overwrite data not yet read).
 * delays_ns is a DEVICE array of len uint32 owned by the caller; it must stay
 * valid while calls that use it run.  len == 0 disarms.
 */
sfar_status sfar_test_set_straggler(sfar_t *h, const uint32_t *delays_ns, uint32_t len, int rank, int phase,
                                    sfar_stream_t s);

/* Rank `rank` (or none if rank < 0) skips every send from the next call on,
 * so its peers' waits run out: the negative test of the bounded waits. */
sfar_status sfar_test_drop_rank(sfar_t *h, int rank, sfar_stream_t s);

/* Wait limit of every device poll, in nanoseconds (default 1 s, or the
 * environment variable SFAR_TIMEOUT_US read by sfar_create). */
sfar_status sfar_test_set_timeout(sfar_t *h, uint64_t ns, sfar_stream_t s);

/* Use parity 0 for every call of the double-buffered protocols (DB, LL,
 * LL128, SENTINEL, TWOSHOT): the negative test of double buffering. */
sfar_status sfar_test_force_single_buffer(sfar_t *h, int on, sfar_stream_t s);

/*
 * Launch mode.  SFAR_LAUNCH_SERIAL (default): stream order.  The kernel is
 * launched as a programmatic dependent of the previous kernel on the stream
 * and waits (griddepcontrol.wait) for it to complete before touching memory,
 * so the end of each kernel is still a full barrier between calls; only the
 * launch overlaps.  SFAR_LAUNCH_PLAIN: stream order with no programmatic
 * launch at all (for comparison).  SFAR_LAUNCH_OVERLAP: each CTA lets the
 * next call's kernel start as soon as it has taken its epoch, and the next
 * call's CTA (r, k) waits only for CTA (r, k) of this call (a wait inside one
 * rank, not across ranks).  Calls may then overtake one another across
 * ranks, which is what double buffering has to survive.  Use OVERLAP only
 * for chains of calls whose inputs do not depend on the previous call's
 * outputs.  In every mode but the cooperative one, a fused AllReduce +
 * RMSNorm call whose grid takes more than three quarters of the device's
 * co-resident clusters runs solo: without programmatic launch, letting no
 * successor launch before it ends.  Every two-shot fused call runs with
 * serial semantics.
 * SFAR_LAUNCH_COOPERATIVE: as SFAR_LAUNCH_SERIAL, and every AllReduce
 * kernel (sfar_allreduce, sfar_allreduce_add_rmsnorm) is launched as a
 * cooperative grid, so the device places it whole (or the call returns
 * SFAR_ERR_UNSUPPORTED when the grid could never be resident) instead of a
 * partly placed grid's waits timing out, and no fused grid runs solo.  It
 * costs the one-shot LL kernel 0.05-0.17 us per call and gains the fused
 * call of four rows of 8192 0.9 us.  Do not profile this mode with Nsight
 * Compute: its replay of a cooperative cluster grid ran the grid without its
 * clusters (the fused kernels then record SFAR_ERR_UNSUPPORTED and run
 * nothing).
 */
#define SFAR_LAUNCH_SERIAL 0
#define SFAR_LAUNCH_OVERLAP 1
#define SFAR_LAUNCH_PLAIN 2
#define SFAR_LAUNCH_COOPERATIVE 3
sfar_status sfar_set_launch_mode(sfar_t *h, int mode);

/*
 * Tracing.  Calls made after this (it is a kernel argument: a captured graph
 * keeps the setting it was captured with) have thread 0 of every CTA write
 * %globaltimer nanoseconds into a ring: entry (e mod calls) of CTA b is
 * trace[((e mod calls) * grid + b) * 8 + point], e the CTA's epoch and grid
 * R * CTAs per rank of that call.  Points: 0 kernel entry, 1 programmatic
 * launch wait returned, 2 epoch known (overlap mode: after the hand-off),
 * 3 first input vector arrived (SFAR_TWOSHOT_TMA: the CTA's tiles are all
 * folded and stored), 4 sends issued (DB/baseline: top barrier passed;
 * SFAR_TWOSHOT_TMA: every rank arrived), 5 receive and reduction done
 * (SFAR_TWOSHOT_TMA: every owner completed), 6 exit; slot 7 holds e itself.
 * trace is a DEVICE array of calls * grid * 8 uint64 owned by the caller;
 * NULL or calls == 0 disarms.
 */
sfar_status sfar_test_set_trace(sfar_t *h, uint64_t *trace, uint32_t calls);

/* Launch geometry of every later call of the receive-buffer protocols:
 * CTAs per rank (0 = automatic; clamped to what can be co-resident) and
 * threads per CTA (0 = automatic, else 64, 128 or 256; the TMA path always
 * uses 320).  SFAR_ERR_INVALID for another thread count.  The fused
 * normalisation calls choose their own shape and ignore this. */
sfar_status sfar_test_set_geometry(sfar_t *h, int ctas_per_rank, int threads_per_cta);

/* Launch shape of sfar_allreduce_add_rmsnorm (allreduce = 1) or
 * sfar_add_rmsnorm (allreduce = 0) for rows x hidden: CTAs per rank, CTAs per
 * thread-block cluster (a row is spread over one cluster) and threads per
 * CTA, of whichever kernel the call would launch (see
 * sfar_test_query_fused_path).  Returns what the call itself would return
 * for the shape (SFAR_ERR_INVALID, SFAR_ERR_UNSUPPORTED) without launching
 * anything. */
sfar_status sfar_test_query_norm_launch(sfar_t *h, size_t rows, size_t hidden, int allreduce, int *ctas_per_rank,
                                        int *cluster_size, int *threads_per_cta);

/* Kernel of every later sfar_allreduce_add_rmsnorm call: path 0 = chosen by
 * shape (default), 1 = the one-shot kernel over LL packets, 2 = the two-shot
 * kernel (each row reduced once by an owner cluster that normalises it for
 * every rank; rows of at most 32 KB whose grid can be resident at once,
 * other shapes keep path 1).
 * SFAR_ERR_INVALID for another value.  Host-side; no launch. */
sfar_status sfar_test_set_fused_path(sfar_t *h, int path);

/* Which kernel sfar_allreduce_add_rmsnorm would launch for rows x hidden
 * under the current setting: *path = 1 (one-shot) or 2 (two-shot).  Returns
 * what the call would return for the shape, without launching anything. */
sfar_status sfar_test_query_fused_path(sfar_t *h, size_t rows, size_t hidden, int *path);

/* Records in sfar_allreduce_noalloc's status block on the current device a
 * wait that gave up (SFAR_ERR_TIMEOUT, the given rank, peer and where code),
 * exactly as a device wait that runs out would: the host-side stand-in for a
 * lost message, to test what callers of that entry point see afterwards.
 * Synchronous; sets the fixed array up first if no call has done so yet. */
sfar_status sfar_test_noalloc_record_failure(int rank, int peer, int where);

/*
 * Latency floor probes.
 * sfar_probe_empty: enqueue one empty kernel (1 CTA, 32 threads) on s.
 * sfar_probe_pingpong: enqueue one kernel of partner + 1 CTAs, one per SM;
 *   CTA 0 and CTA `partner` (1 <= partner < SM count) pass a token `trips`
 *   times through two flags in global memory (relaxed == 0: st.release /
 *   ld.acquire at GPU scope; relaxed != 0: relaxed GPU-scope stores and
 *   loads).  out (device, 3 uint64) gets the elapsed %globaltimer
 *   nanoseconds and the SM ids of the two CTAs; which SMs they land on
 *   decides the round trip (on the same die or across dies), so callers
 *   sweep `partner`.  flags is a device array of 64 uint32 that the probe
 *   zeroes first.  Waits are bounded (1 s); on timeout out[0] = UINT64_MAX.
 */
sfar_status sfar_probe_empty(sfar_stream_t s);
sfar_status sfar_probe_pingpong(uint32_t *flags, int trips, int relaxed, int partner, uint64_t *out,
                                sfar_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* SFAR_TEST_H */
