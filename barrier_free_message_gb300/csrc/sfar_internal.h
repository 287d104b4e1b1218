// sfar_internal.h -- layout shared by the host code and the kernels of libsfar.
#pragma once
#include <stddef.h>
#include <stdint.h>

#define SFAR_MAX_R 16
#define SFAR_KMAX 128                       // CTAs per rank, upper bound (flag array stride)
#define SFAR_THREADS 256                    // threads per CTA of the receive-buffer kernels
#define SFAR_WARPS (SFAR_THREADS / 32)
#define SFAR_RECV_MAX_BYTES (2ull << 20)    // per-rank limit of the receive-buffer protocols
#define SFAR_LL128_PAYLOAD 124              // bytes of payload per 128-byte LL128 line
#define SFAR_ITER_BYTES (4 * SFAR_LL128_PAYLOAD)   // payload of the 4 lines one warp moves at once
#define SFAR_TMA_THREADS 320                // TMA path: 8 consumer warps, a producer and a store warp
#define SFAR_NTHREAD_OPTS 3                 // receive-buffer kernels: 64, 128 or 256 threads
#define SFAR_LL_UNIT_NARROW 8               // LL kernel: input bytes per thread for R <= 8 (16, 8 or 4)
#define SFAR_LL_UNIT_WIDE 8                 // and for R > 8
#define SFAR_SENT_UNIT 8                    // sentinel kernel: input bytes per thread (16 or 8)
#define SFAR_FLAG_STRIDE 1                  // u32 words between the flags of consecutive CTA indices
// Arrival and completion flags of the pull protocols (TMA AllReduce, two-shot
// fused normalisation): one 128-byte line per flag.  Packed, the flags of the
// up to 128 CTAs of a rank shared a few lines that every CTA of every peer
// polls; spread out, a two-shot fused call of 64 rows of 7168 at R = 8 passed
// its arrival barrier in 2.6 instead of 5.4 us (24.9 -> 21.3 us per call),
// and the TMA AllReduce at 1 MB per rank took 10.0 instead of 10.8 us.  The
// ready flags of DB and BASELINE stay packed (3% faster that way).
#define SFAR_PULL_FLAG_STRIDE 32

// Index of the flag of CTA index k in row `row` of a flag array laid out
// [rows][SFAR_KMAX] with SFAR_FLAG_STRIDE (or, for the pull protocols,
// SFAR_PULL_FLAG_STRIDE) words per flag.
#ifdef __CUDACC__
__host__ __device__
#endif
inline size_t sfar_flag(size_t row, int k)
{
    return (row * SFAR_KMAX + (size_t)k) * SFAR_FLAG_STRIDE;
}
#ifdef __CUDACC__
__host__ __device__
#endif
inline size_t sfar_pull_flag(size_t row, int k)
{
    return (row * SFAR_KMAX + (size_t)k) * SFAR_PULL_FLAG_STRIDE;
}

// Device status block of one handle.  The first 32 bytes are the sticky
// status and the fault record; the knobs follow.
struct SfarCtl {
    int status;               // 0 = OK, else SFAR_ERR_TIMEOUT (sticky until reset)
    int f_rank, f_cta, f_peer;
    uint32_t f_epoch;
    int f_where;
    int pad0[2];
    unsigned long long timeout_ns;
    // knobs, read only by the test variants of the kernels
    const uint32_t *strag_delays;
    uint32_t strag_len;
    int strag_rank;           // < 0: rotating (call mod R)
    int strag_phase;          // 0: before the sends, 1: between sends and receives
    int drop_rank;            // < 0: none
    int single_buffer;
    uint32_t strag_base;              // last epoch when the straggler was armed
};
#define SFAR_TRACE_POINTS 8

// Kernel parameters, passed by value (fits the parameter space).
struct SfarArgs {
    const void *in[SFAR_MAX_R];
    void *out[SFAR_MAX_R];
    unsigned long long n;         // elements per rank
    unsigned long long slot;      // bytes per (receiver, parity, sender) slot of `region`
    unsigned long long chunk;     // two-shot: elements per owner chunk
    unsigned long long sub;       // TMA path: elements per CTA range within a chunk
    uint8_t *region;              // receive region of the protocol (atomic path: accumulator lines)
    uint8_t *region2;             // two-shot and atomic path: all-gather region
    unsigned long long *epoch;    // [R] call counters: + SFAR_KMAX per call (see the prologue)
    uint32_t *done;               // [R][SFAR_KMAX] last finished epoch (overlap mode)
    uint32_t *fa;                 // flags [R][R][SFAR_KMAX]: ready / top barrier / arrival
    uint32_t *fb;                 // flags [R][R][SFAR_KMAX]: bottom barrier / completion
    SfarCtl *ctl;
    int R, K, overlap, tile_bytes, stages;
    unsigned long long *trace;    // NULL, or a ring of trace_calls entries per CTA (see sfar_test.h)
    uint32_t trace_calls;
    int solo;                     // 1: launched without overlap, and lets no successor launch early
};

// Kernel lookup, one function per translation unit.  dt: 0 bf16, 1 fp32.
// wide: R > 8.  test: the variant that reads the knobs.
const void *sfar_kernel_ll(int dt, int wide, int test);
const void *sfar_kernel_ll128(int dt, int wide, int test);
const void *sfar_kernel_sentinel(int dt, int wide, int test);
const void *sfar_kernel_db(int dt, int wide, int test, int baseline);
const void *sfar_kernel_twoshot(int dt, int wide, int test);
const void *sfar_kernel_twoshot_sent(int dt, int wide, int test);
const void *sfar_kernel_tma(int dt, int test);
const void *sfar_kernel_atomic(int dt, int wide, int test);
const void *sfar_kernel_set_knob();
const void *sfar_kernel_empty();
const void *sfar_kernel_pingpong();

// Knob writes (one-thread kernel): which field and value.
enum SfarKnob {
    KNOB_TIMEOUT = 1,
    KNOB_STRAG = 2,
    KNOB_DROP = 3,
    KNOB_SINGLE = 4,
    KNOB_CLEAR_STATUS = 5
};
struct SfarKnobArgs {
    SfarCtl *ctl;
    int which;
    unsigned long long value;
    const uint32_t *ptr;
    uint32_t len;
    int rank;
    int phase;
    const unsigned long long *epoch0;   // rank 0's call counter, for the straggler base
};
