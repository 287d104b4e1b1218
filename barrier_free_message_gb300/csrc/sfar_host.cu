// sfar_host.cu -- the C ABI of libsfar: handle, buffers, launch, status.
//
// The handle is the analogue of the pages' LLBuffer object ("Every
// Microsecond Counts" (page 1), section "Unified primitives and API design":
// a buffer object that hides the slot layout, the synchronisation mode, the
// epoch and the reset).  One device allocation holds, for R simulated ranks,
// the receive regions of every protocol, the flags, the per-(rank, CTA)
// epoch counters and the status block ("symmetric memory" of the pages
// becomes regions at fixed offsets of one allocation).  A call validates its
// arguments on the host and enqueues exactly one kernel; nothing is
// allocated or synchronised per call, so calls can be captured in a CUDA
// graph and replayed with no host involvement (the epochs live on the device).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "sfar.h"
#include "sfar_decode.h"
#include "sfar_fused.h"
#include "sfar_gemv.h"
#include "sfar_internal.h"
#include "sfar_test.h"

namespace {

thread_local sfar_status g_last_error = SFAR_OK;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
size_t ceil_div(size_t x, size_t a) { return (x + a - 1) / a; }

// TMA path: each CTA takes at least this many bytes of a chunk, so from
// about 150 KB per chunk every SM streams (one CTA per SM).
const size_t kTmaMinBytesPerCta = 8u << 10;

}  // namespace

struct sfar {
    int R = 0;
    size_t max_bytes = 0;
    int dt = 0, es = 2;
    int dev = 0, sms = 0;
    size_t rb = 0;                      // per-rank limit of the receive-buffer protocols
    uint8_t *ws = nullptr;
    size_t ws_bytes = 0;
    size_t ctl_bytes = 0;               // the status block sits at the start of ws
    unsigned long long *epoch = nullptr;   // [R] per-rank call counters
    uint32_t *done = nullptr;
    uint32_t *fa = nullptr, *fb = nullptr, *fc = nullptr, *fd = nullptr;
    SfarCtl *ctl = nullptr;
    uint8_t *r_raw = nullptr, *r_ll = nullptr, *r_ll128 = nullptr, *r_sent = nullptr;
    uint8_t *r_rs = nullptr, *r_ag = nullptr;
    uint8_t *r_srs = nullptr, *r_sag = nullptr;   // sentinel two-shot: RS and AG regions (sentinel-prefilled)
    uint8_t *r_acc = nullptr, *r_agx = nullptr;   // atomic path: accumulator and all-gather lines
    size_t s_raw = 0, s_ll = 0, s_ll128 = 0, s_2s = 0, s_at = 0, s_ts = 0, sent_bytes = 0;
    int mode = SFAR_LAUNCH_SERIAL;
    int ctas_override = 0, threads_override = 0;
    long long last_key = -1;            // overlap mode: geometry of the previous call
    sfar_stream_t last_stream = nullptr;
    unsigned long long last_capture = 0;
    unsigned long long *trace = nullptr; // test hook: trace ring (device), calls per CTA
    uint32_t trace_calls = 0;
    bool k_strag = false, k_drop = false, k_single = false;
    bool poisoned = false;
    cudaStream_t priv = nullptr;
    SfarCtl *host_ctl = nullptr;
    int kmax[SFAR_NUM_PROTOS][SFAR_NTHREAD_OPTS] = {};   // co-resident CTAs per rank
    int tma_tb = 0, tma_ns = 0;
    size_t tma_smem = 0;
    // fused normalisation: co-resident clusters per launch shape, queried once
    // ([allreduce][test][batched][8-byte units][cluster size][threads index], 0 = not yet known)
    int norm_clusters[2][2][2][2][SFAR_NORM_CLMAX + 1][4] = {};
    // two-shot fused kernel: co-resident clusters ([test][cluster size][threads index])
    int ts_clusters[2][SFAR_NORM_CLMAX + 1][4] = {};
    int fused_path = 0;                 // test knob: 0 by shape, 1 one-shot LL, 2 two-shot
};

static const void *kernel_for(const sfar *h, int p, int test)
{
    const int wide = h->R > 8;
    switch (p) {
    case SFAR_BASELINE: return sfar_kernel_db(h->dt, wide, test, 1);
    case SFAR_DB: return sfar_kernel_db(h->dt, wide, test, 0);
    case SFAR_LL: return sfar_kernel_ll(h->dt, wide, test);
    case SFAR_LL128: return sfar_kernel_ll128(h->dt, wide, test);
    case SFAR_SENTINEL: return sfar_kernel_sentinel(h->dt, wide, test);
    case SFAR_TWOSHOT: return sfar_kernel_twoshot(h->dt, wide, test);
    case SFAR_TWOSHOT_SENTINEL: return sfar_kernel_twoshot_sent(h->dt, wide, test);
    case SFAR_TWOSHOT_TMA: return sfar_kernel_tma(h->dt, test);
    case SFAR_LL128_ATOMIC: return sfar_kernel_atomic(h->dt, wide, test);
    default: return nullptr;
    }
}

static size_t smem_for(const sfar *h, int p) { return p == SFAR_TWOSHOT_TMA ? h->tma_smem : 0; }

// Thread counts a receive-buffer kernel may be launched with (index ti).
static const int kThreadOpts[SFAR_NTHREAD_OPTS] = {64, 128, 256};

static int thread_index(int threads)
{
    for (int i = 0; i < SFAR_NTHREAD_OPTS; ++i)
        if (kThreadOpts[i] == threads)
            return i;
    return -1;
}

// Work units of a call: 16-byte vectors (one-shot vector protocols; the LL
// kernel's unit for LL), 4-line groups per warp (LL128, two-shot), lines of a
// chunk per warp (atomic path), or bytes of a chunk (TMA path).
static size_t work_units(const sfar *h, int p, size_t n, size_t *chunk)
{
    const size_t nvec = ceil_div(n * (size_t)h->es, 16);
    *chunk = 0;
    switch (p) {
    case SFAR_LL:
        return ceil_div(n * (size_t)h->es, h->R > 8 ? SFAR_LL_UNIT_WIDE : SFAR_LL_UNIT_NARROW);
    case SFAR_SENTINEL:
        return ceil_div(n * (size_t)h->es, SFAR_SENT_UNIT);
    case SFAR_LL128:
        return ceil_div(nvec, 31);
    case SFAR_TWOSHOT: {
        const size_t epi = SFAR_ITER_BYTES / (size_t)h->es;   // elements per 4-line group
        *chunk = align_up(ceil_div(n, (size_t)h->R), epi);
        return *chunk / epi;
    }
    case SFAR_TWOSHOT_TMA:
        *chunk = align_up(ceil_div(n, (size_t)h->R), 16 / (size_t)h->es);
        return *chunk * (size_t)h->es;
    case SFAR_TWOSHOT_SENTINEL:                                // 8-byte units of a chunk
        *chunk = align_up(ceil_div(n, (size_t)h->R), 16 / (size_t)h->es);
        return *chunk * (size_t)h->es / 8;
    case SFAR_LL128_ATOMIC:
        *chunk = align_up(ceil_div(n, (size_t)h->R), 31);
        return *chunk / 31;
    default:
        return nvec;
    }
}

// Launch geometry: CTAs per rank (K), threads per CTA and, for the chunked
// paths, chunk and per-CTA range in elements.  Without an override, the
// receive-buffer kernels take the smallest CTA that keeps one work unit per
// thread (or per warp) while the whole grid fits on the SMs once, so the
// R * K CTAs spread over as many SMs as the message can use.
static int geometry(const sfar *h, int p, size_t n, size_t *chunk, size_t *sub, int *threads)
{
    const size_t units = work_units(h, p, n, chunk);
    *sub = 0;
    const bool warp_units = p == SFAR_LL128 || p == SFAR_TWOSHOT || p == SFAR_LL128_ATOMIC;
    int ti = SFAR_NTHREAD_OPTS - 1;
    size_t K = 1;
    if (p == SFAR_TWOSHOT_TMA) {
        *threads = SFAR_TMA_THREADS;
        ti = 0;
        K = ceil_div(units, kTmaMinBytesPerCta);
    } else {
        if (h->threads_override > 0 && thread_index(h->threads_override) >= 0) {
            ti = thread_index(h->threads_override);
        } else {
            // the flag protocols pay per CTA for their barrier, so they start at 128 threads
            const int first = (p == SFAR_DB || p == SFAR_BASELINE) ? 1 : 0;
            for (int i = first; i < SFAR_NTHREAD_OPTS; ++i) {
                const size_t per = warp_units ? (size_t)kThreadOpts[i] / 32 : (size_t)kThreadOpts[i];
                if ((size_t)h->R * ceil_div(units, per) <= (size_t)h->sms) {
                    ti = i;
                    break;
                }
            }
        }
        *threads = kThreadOpts[ti];
        const size_t per = warp_units ? (size_t)*threads / 32 : (size_t)*threads;
        K = ceil_div(units, per);
    }
    if (h->ctas_override > 0)
        K = (size_t)h->ctas_override;
    if (K < 1)
        K = 1;
    if (K > (size_t)h->kmax[p][ti])
        K = (size_t)h->kmax[p][ti];
    // TMA path: one CTA per SM, so that the next call's CTAs, launched early,
    // find room beside this call's (two fit by shared memory from R = 4)
    if (p == SFAR_TWOSHOT_TMA && K > (size_t)h->sms / (size_t)h->R)
        K = (size_t)h->sms / (size_t)h->R;
    if (p == SFAR_TWOSHOT_TMA)
        *sub = align_up(ceil_div(*chunk, K), 16 / (size_t)h->es);
    return (int)K;
}

static sfar_status launch_knob(sfar *h, int which, unsigned long long value, const uint32_t *ptr, uint32_t len,
                               int rank, cudaStream_t s, int phase = 0)
{
    SfarKnobArgs k;
    memset(&k, 0, sizeof k);
    k.ctl = h->ctl;
    k.which = which;
    k.value = value;
    k.ptr = ptr;
    k.len = len;
    k.rank = rank;
    k.phase = phase;
    k.epoch0 = h->epoch;
    void *args[] = {&k};
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != h->dev)
        cudaSetDevice(h->dev);
    cudaError_t err = cudaLaunchKernel(sfar_kernel_set_knob(), dim3(1), dim3(1), args, 0, s);
    if (cur != h->dev && cur >= 0)
        cudaSetDevice(cur);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    return SFAR_OK;
}

extern "C" {

sfar_status sfar_last_error(void) { return g_last_error; }

const char *sfar_strerror(sfar_status st)
{
    switch (st) {
    case SFAR_OK: return "ok";
    case SFAR_ERR_INVALID: return "invalid argument";
    case SFAR_ERR_CUDA: return "CUDA runtime error";
    case SFAR_ERR_OOM: return "out of memory";
    case SFAR_ERR_TIMEOUT: return "a bounded device wait gave up (lost message or stalled rank)";
    case SFAR_ERR_UNSUPPORTED: return "unsupported device or launch geometry";
    case SFAR_ERR_POISONED: return "handle poisoned by an earlier device failure; call sfar_reset";
    default: return "unknown status";
    }
}

sfar_t *sfar_create(int R, size_t max_bytes, sfar_dtype dt)
{
    if (R < 2 || R > SFAR_MAX_R || max_bytes == 0 || (dt != SFAR_BF16 && dt != SFAR_FP32)) {
        g_last_error = SFAR_ERR_INVALID;
        return nullptr;
    }
    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        g_last_error = SFAR_ERR_CUDA;
        return nullptr;
    }
    if (major != 10 || minor != 3) {
        g_last_error = SFAR_ERR_UNSUPPORTED;
        return nullptr;
    }
    sfar *h = new (std::nothrow) sfar();
    if (!h) {
        g_last_error = SFAR_ERR_OOM;
        return nullptr;
    }
    h->R = R;
    h->max_bytes = max_bytes;
    h->dt = (int)dt;
    h->es = dt == SFAR_BF16 ? 2 : 4;
    h->dev = dev;
    h->sms = sms;
    h->rb = align_up(max_bytes < SFAR_RECV_MAX_BYTES ? max_bytes : SFAR_RECV_MAX_BYTES, 16);

    // slot sizes (bytes per receiver, parity, sender)
    const size_t nvec = h->rb / 16;
    h->s_raw = align_up(h->rb, 256);
    h->s_ll = align_up(2 * h->rb, 256);
    h->s_ll128 = align_up(ceil_div(nvec, 31) * 512, 256);
    {
        const size_t nmax = h->rb / (size_t)h->es;
        const size_t epi = SFAR_ITER_BYTES / (size_t)h->es;
        const size_t c = align_up(ceil_div(nmax, (size_t)R), epi);
        h->s_2s = align_up(c / epi * 512, 256);
        // atomic path: 128-byte lines of 31 elements per (owner, parity)
        h->s_at = align_up(ceil_div(ceil_div(nmax, (size_t)R), 31) * 128, 256);
        // sentinel two-shot: one chunk of raw bytes per (owner or receiver, parity, peer)
        h->s_ts = align_up(align_up(ceil_div(nmax, (size_t)R), 16 / (size_t)h->es) * (size_t)h->es, 256);
    }
    const size_t RR2 = (size_t)R * 2 * R;
    size_t off = 0;
    auto carve = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    const size_t o_ctl = carve(sizeof(SfarCtl));
    h->ctl_bytes = off;
    const size_t o_epoch = carve((size_t)R * sizeof(unsigned long long));
    const size_t o_done = carve((size_t)R * SFAR_KMAX * 4);
    const size_t o_fa = carve((size_t)R * R * SFAR_KMAX * SFAR_FLAG_STRIDE * 4);
    const size_t o_fb = carve((size_t)R * R * SFAR_KMAX * SFAR_FLAG_STRIDE * 4);
    const size_t o_fc = carve((size_t)R * SFAR_KMAX * SFAR_PULL_FLAG_STRIDE * 4);
    const size_t o_fd = carve((size_t)R * R * SFAR_KMAX * SFAR_PULL_FLAG_STRIDE * 4);
    const size_t o_raw = carve(RR2 * h->s_raw);
    const size_t o_ll = carve(RR2 * h->s_ll);
    const size_t o_ll128 = carve(RR2 * h->s_ll128);
    const size_t o_rs = carve(RR2 * h->s_2s);
    const size_t o_ag = carve(RR2 * h->s_2s);
    const size_t o_sent = carve(RR2 * h->s_raw);            // the sentinel-prefilled regions, back to back
    const size_t o_srs = carve(RR2 * h->s_ts);
    const size_t o_sag = carve(RR2 * h->s_ts);
    const size_t o_acc = carve((size_t)R * 2 * h->s_at);
    const size_t o_agx = carve(RR2 * h->s_at);
    h->sent_bytes = o_sag + RR2 * h->s_ts - o_sent;
    h->ws_bytes = off;

    if (cudaMalloc(&h->ws, h->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        g_last_error = SFAR_ERR_OOM;
        return nullptr;
    }
    h->ctl = reinterpret_cast<SfarCtl *>(h->ws + o_ctl);
    h->epoch = reinterpret_cast<unsigned long long *>(h->ws + o_epoch);
    h->done = reinterpret_cast<uint32_t *>(h->ws + o_done);
    h->fa = reinterpret_cast<uint32_t *>(h->ws + o_fa);
    h->fb = reinterpret_cast<uint32_t *>(h->ws + o_fb);
    h->fc = reinterpret_cast<uint32_t *>(h->ws + o_fc);
    h->fd = reinterpret_cast<uint32_t *>(h->ws + o_fd);
    h->r_raw = h->ws + o_raw;
    h->r_ll = h->ws + o_ll;
    h->r_ll128 = h->ws + o_ll128;
    h->r_rs = h->ws + o_rs;
    h->r_ag = h->ws + o_ag;
    h->r_sent = h->ws + o_sent;
    h->r_srs = h->ws + o_srs;
    h->r_sag = h->ws + o_sag;
    h->r_acc = h->ws + o_acc;
    h->r_agx = h->ws + o_agx;

    // TMA path: a stage holds R tiles (about 48 KB in all, 32 KB at R = 2);
    // as many stages as keep about 96 KB of input tiles in flight per SM, at
    // least 2.  Measured against filling 220 KB of shared memory (R = 2 to
    // 16, 16-256 MB per rank): 2-4 stages of about 48 KB beat 3-5 (R = 8,
    // 64 MB: 0.915 -> 0.947 of the copy bandwidth; R = 16: 0.897 -> 0.982),
    // and at R = 2 three stages of 32 KB beat two and five.
    {
        size_t tb = 49152 / (size_t)R;
        if (tb < 2048) tb = 2048;
        if (tb > 16384) tb = 16384;
        tb &= ~(size_t)15;
        const size_t in_flight = 96u << 10, outb = 3 * tb;
        size_t ns = in_flight / ((size_t)R * tb);
        if (ns < 2) ns = 2;
        if (ns > 8) ns = 8;
        h->tma_tb = (int)tb;
        h->tma_ns = (int)ns;
        h->tma_smem = ns * R * tb + outb + (2 * ns + 2 * 3) * 8;   // + full/empty and buffer mbarriers
    }

    SfarCtl init;
    memset(&init, 0, sizeof init);
    unsigned long long timeout_ns = 1000000000ull;
    if (const char *env = getenv("SFAR_TIMEOUT_US")) {
        const unsigned long long us = strtoull(env, nullptr, 10);
        if (us > 0)
            timeout_ns = us * 1000ull;
    }
    init.timeout_ns = timeout_ns;
    init.strag_rank = -1;
    init.drop_rank = -1;
    init.f_rank = init.f_cta = init.f_peer = -1;

    sfar_status st = SFAR_OK;
    if (cudaMemset(h->ws, 0, h->ws_bytes) != cudaSuccess || cudaMemset(h->r_sent, 0xff, h->sent_bytes) != cudaSuccess ||
        cudaMemcpy(h->ctl, &init, sizeof init, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h->priv, cudaStreamNonBlocking) != cudaSuccess ||
        cudaMallocHost(&h->host_ctl, sizeof(SfarCtl)) != cudaSuccess)
        st = SFAR_ERR_CUDA;
    for (int test = 0; test < 2 && st == SFAR_OK; ++test) {
        const void *f = kernel_for(h, SFAR_TWOSHOT_TMA, test);
        if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)h->tma_smem) != cudaSuccess)
            st = SFAR_ERR_UNSUPPORTED;
    }
    if (st == SFAR_OK &&
        cudaFuncSetAttribute(sfar_kernel_gemv(), cudaFuncAttributeMaxDynamicSharedMemorySize, SFAR_GEMV_SMEM) !=
            cudaSuccess)
        st = SFAR_ERR_UNSUPPORTED;
    // co-residency: every CTA of a call must be resident at once (ranks wait
    // on each other), so K is capped by the occupancy of each variant
    for (int p = 0; p < SFAR_NUM_PROTOS && st == SFAR_OK; ++p) {
        const int nopts = p == SFAR_TWOSHOT_TMA ? 1 : SFAR_NTHREAD_OPTS;
        for (int ti = 0; ti < nopts && st == SFAR_OK; ++ti) {
            const int threads = p == SFAR_TWOSHOT_TMA ? SFAR_TMA_THREADS : kThreadOpts[ti];
            int km = SFAR_KMAX;
            for (int test = 0; test < 2; ++test) {
                int nb = 0;
                if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kernel_for(h, p, test), threads,
                                                                  smem_for(h, p)) != cudaSuccess) {
                    st = SFAR_ERR_CUDA;
                    break;
                }
                const int k = nb * sms / R;
                if (k < km)
                    km = k;
            }
            if (km < 1)
                st = SFAR_ERR_UNSUPPORTED;
            h->kmax[p][ti] = km;
        }
    }
    if (st == SFAR_OK && cudaDeviceSynchronize() != cudaSuccess)
        st = SFAR_ERR_CUDA;
    if (st != SFAR_OK) {
        cudaGetLastError();
        sfar_destroy(h);
        g_last_error = st;
        return nullptr;
    }
    g_last_error = SFAR_OK;
    return h;
}

void sfar_destroy(sfar_t *h)
{
    if (!h)
        return;
    if (h->ws)
        cudaFree(h->ws);
    if (h->host_ctl)
        cudaFreeHost(h->host_ctl);
    if (h->priv)
        cudaStreamDestroy(h->priv);
    delete h;
}

size_t sfar_max_bytes(const sfar_t *h, sfar_proto p)
{
    if (!h || (int)p < 0 || (int)p >= SFAR_NUM_PROTOS)
        return 0;
    return p == SFAR_TWOSHOT_TMA ? h->max_bytes : h->rb;
}

sfar_status sfar_query_launch(const sfar_t *h, size_t n, sfar_proto p, int *ctas_per_rank, int *threads_per_cta)
{
    if (!h || (int)p < 0 || (int)p >= SFAR_NUM_PROTOS)
        return SFAR_ERR_INVALID;
    size_t chunk, sub;
    int threads = 0;
    const int K = geometry(h, p, n, &chunk, &sub, &threads);
    if (ctas_per_rank)
        *ctas_per_rank = K;
    if (threads_per_cta)
        *threads_per_cta = threads;
    return SFAR_OK;
}

sfar_status sfar_allreduce(sfar_t *h, const void *const in[], void *const out[], size_t n, sfar_proto p,
                           sfar_stream_t s)
{
    if (!h || (int)p < 0 || (int)p >= SFAR_NUM_PROTOS)
        return SFAR_ERR_INVALID;
    if (h->poisoned)
        return SFAR_ERR_POISONED;
    if (n == 0)
        return SFAR_OK;
    if (!in || !out || n > ((size_t)-1) / 16)
        return SFAR_ERR_INVALID;
    const int R = h->R;
    const size_t bytes = n * (size_t)h->es;
    if (bytes > sfar_max_bytes(h, p))
        return SFAR_ERR_INVALID;
    for (int r = 0; r < R; ++r) {
        if (!in[r] || !out[r] || ((uintptr_t)in[r] & 15u) || ((uintptr_t)out[r] & 15u))
            return SFAR_ERR_INVALID;
    }
    // no output may overlap an input or another output
    for (int i = 0; i < R; ++i) {
        const uintptr_t o0 = (uintptr_t)out[i], o1 = o0 + bytes;
        for (int j = 0; j < R; ++j) {
            const uintptr_t a0 = (uintptr_t)in[j], a1 = a0 + bytes;
            if (o0 < a1 && a0 < o1)
                return SFAR_ERR_INVALID;
            if (j != i) {
                const uintptr_t b0 = (uintptr_t)out[j], b1 = b0 + bytes;
                if (o0 < b1 && b0 < o1)
                    return SFAR_ERR_INVALID;
            }
        }
    }

    SfarArgs a;
    memset(&a, 0, sizeof a);
    for (int r = 0; r < R; ++r) {
        a.in[r] = in[r];
        a.out[r] = out[r];
    }
    size_t chunk = 0, sub = 0;
    int threads = 0;
    const int K = geometry(h, p, n, &chunk, &sub, &threads);
    a.n = n;
    a.chunk = chunk;
    a.sub = sub;
    a.epoch = h->epoch;
    a.done = h->done;
    a.ctl = h->ctl;
    a.R = R;
    a.K = K;
    // Overlap mode lets a call overtake the previous one only when the two
    // run the same kernel geometry on the same stream (the hand-off is between
    // CTAs of the same index); the first call of a graph capture, or one after
    // a change, is launched with serial semantics.
    a.overlap = 0;
    if (h->mode == SFAR_LAUNCH_OVERLAP) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        unsigned long long cap = 0;
        if (cudaStreamGetCaptureInfo((cudaStream_t)s, &cs, &cap) != cudaSuccess) {
            cudaGetLastError();
            cs = cudaStreamCaptureStatusNone;
        }
        if (cs != cudaStreamCaptureStatusActive)
            cap = 0;
        const long long key = ((long long)p << 40) | ((long long)K << 16) | threads;
        a.overlap = (key == h->last_key && s == h->last_stream && cap == h->last_capture) ? 1 : 0;
        h->last_key = key;
        h->last_stream = s;
        h->last_capture = cap;
    }
    a.trace = h->trace;
    a.trace_calls = h->trace_calls;
    switch (p) {
    case SFAR_BASELINE:
    case SFAR_DB:
        a.region = h->r_raw;
        a.slot = h->s_raw;
        a.fa = h->fa;
        a.fb = h->fb;
        break;
    case SFAR_LL:
        a.region = h->r_ll;
        a.slot = h->s_ll;
        break;
    case SFAR_LL128:
        a.region = h->r_ll128;
        a.slot = h->s_ll128;
        break;
    case SFAR_SENTINEL:
        a.region = h->r_sent;
        a.slot = h->s_raw;
        break;
    case SFAR_TWOSHOT:
        a.region = h->r_rs;
        a.region2 = h->r_ag;
        a.slot = h->s_2s;
        break;
    case SFAR_LL128_ATOMIC:
        a.region = h->r_acc;
        a.region2 = h->r_agx;
        a.slot = h->s_at;
        break;
    case SFAR_TWOSHOT_SENTINEL:
        a.region = h->r_srs;
        a.region2 = h->r_sag;
        a.slot = h->s_ts;
        break;
    case SFAR_TWOSHOT_TMA:
        a.fa = h->fc;
        a.fb = h->fd;
        a.tile_bytes = h->tma_tb;
        a.stages = h->tma_ns;
        break;
    }
    const int test = (h->k_strag || h->k_drop || h->k_single) ? 1 : 0;

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(R * K));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem_for(h, p);
    cfg.stream = (cudaStream_t)s;
    cudaLaunchAttribute attr[2];
    int nattr = 0;
    if (h->mode != SFAR_LAUNCH_PLAIN) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    if (h->mode == SFAR_LAUNCH_COOPERATIVE) {
        // every CTA of the grid is placed at once, or the launch fails
        attr[nattr].id = cudaLaunchAttributeCooperative;
        attr[nattr].val.cooperative = 1;
        ++nattr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    void *args[] = {&a};
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != h->dev)
        cudaSetDevice(h->dev);
    cudaError_t err = cudaLaunchKernelExC(&cfg, kernel_for(h, p, test), args);
    if (cur != h->dev && cur >= 0)
        cudaSetDevice(cur);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return err == cudaErrorCooperativeLaunchTooLarge ? SFAR_ERR_UNSUPPORTED : SFAR_ERR_CUDA;
    }
    return SFAR_OK;
}

// ------------------------------------------------- fused AllReduce + RMSNorm
static const int kNormThreads[4] = {32, 64, 128, 256};

// Cluster size and threads for a row of VR units: one unit per thread over
// a cluster of up to 8 CTAs where it fits (*CL) -- 128 threads per CTA up to
// 1024 units, 256 threads beyond for 8-byte units; for 16-byte units 128
// threads up to 4096 units, 256 beyond (up to 8192).  *CLmin is the smallest
// cluster that still gives every thread at most SFAR_NORM_VMAX units.  Rows
// of up to 128 units take one CTA.
static bool norm_shape(unsigned long long VR, int unit, int *CL, int *CLmin, int *ti)
{
    if (VR <= 128) {
        *CL = *CLmin = 1;
        *ti = VR <= 32 ? 0 : VR <= 64 ? 1 : 2;
        return true;
    }
    const int t = VR <= (unit == 8 ? 1024u : 4096u) ? 128 : 256;
    *ti = t == 128 ? 2 : 3;
    int cl = (int)ceil_div(VR, (size_t)t);
    if (cl > SFAR_NORM_CLMAX)
        cl = SFAR_NORM_CLMAX;
    *CL = cl;
    *CLmin = (int)ceil_div(VR, (size_t)t * SFAR_NORM_VMAX);
    return *CLmin <= cl;
}

static int norm_max_clusters(sfar *h, int allreduce, int test, int batch, int unit, int CL, int ti)
{
    int &slot = h->norm_clusters[allreduce][test][batch > 1 ? 1 : 0][unit == 8 ? 1 : 0][CL][ti];
    if (slot)
        return slot;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)CL);
    cfg.blockDim = dim3((unsigned)kNormThreads[ti]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sfar_kernel_fused(h->dt, h->R > 8, allreduce, test, batch, unit), &cfg) !=
        cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    slot = n > 0 ? n : -1;
    return slot;
}

// Except in cooperative mode, a fused AllReduce grid whose clusters take
// more than three quarters of `maxc` (the co-resident clusters that the
// occupancy query reports for an idle device) runs solo: launched without
// programmatic overlap, it starts on an idle device and lets no successor
// launch before it ends.  Cooperative mode launches the grid as a
// cooperative grid instead (see fused_call).  Every CTA of
// such a grid waits on others, and a large cluster grid launched early, while
// its predecessor still held the device, did not always get all of its
// clusters placed: R = 8, eight rows of 8192 bf16, 32 of 36 clusters of 8
// CTAs, timed out on its last rank in 12 of 40 graph replays of 32 calls with
// overlap and in none without.  Grids at 70% and 79% of `maxc` ran thousands
// of overlapped calls without a stall.
static bool solo_grid(int clusters, int maxc) { return 4 * clusters > 3 * maxc; }

// Launch shape of a fused call: threads per CTA, cluster size (shrunk from
// the preferred one while R clusters cannot be resident at once), clusters
// per rank G (K = G * CL <= KMAX), vectors of a row per thread, and rows per
// statistics round (up to 4 when every thread holds one vector of each row
// and a cluster gets more than one row).
static sfar_status norm_geometry(sfar *h, int allreduce, int test, size_t rows, unsigned long long VR, int unit,
                                 int *CL_out, int *G_out, int *threads_out, int *vpt_out, int *batch_out,
                                 int *maxc_out)
{
    int CL = 0, CLmin = 0, ti = 0;
    if (!norm_shape(VR, unit, &CL, &CLmin, &ti))
        return SFAR_ERR_INVALID;
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != h->dev)
        cudaSetDevice(h->dev);
    int maxc = -1, vpt = 1, nb = 1;
    for (; CL >= CLmin; --CL) {
        vpt = (int)ceil_div(VR, (size_t)CL * kNormThreads[ti]);
        nb = (vpt == 1 && rows > 1) ? 4 : 1;
        maxc = norm_max_clusters(h, allreduce, test, nb, unit, CL, ti);
        if (maxc < 0 || maxc >= h->R)
            break;
    }
    if (cur != h->dev && cur >= 0)
        cudaSetDevice(cur);
    if (maxc < 0)
        return SFAR_ERR_CUDA;
    if (CL < CLmin)
        return SFAR_ERR_UNSUPPORTED;
    size_t G = (size_t)maxc / (size_t)h->R;
    if (G > (size_t)(SFAR_KMAX / CL))
        G = (size_t)(SFAR_KMAX / CL);
    if (G > rows)
        G = rows;
    if (G < 1)
        G = 1;
    size_t B = nb;
    if (B > ceil_div(rows, G))
        B = ceil_div(rows, G);                    // no more rows per round than a cluster gets
    *CL_out = CL;
    *G_out = (int)G;
    *maxc_out = maxc;
    *threads_out = kNormThreads[ti];
    *vpt_out = vpt;
    *batch_out = (int)B;
    return SFAR_OK;
}

// Two-shot fused call: a row over one cluster of CL CTAs with one 16-byte
// unit per thread (32-128 threads per CTA; 256 above 1024 units, and above
// 512 units when a rank gets several clusters: fewer, larger CTAs start and
// synchronise sooner there, 4% faster at 16 and 64 rows of 896 units, but 11%
// slower with one cluster per rank; rows of at most 32 KB), and G clusters per rank: as
// many as the rows need, all of the grid resident at once (its CTAs wait on
// one another).
static sfar_status ts_geometry(sfar *h, int test, size_t rows, unsigned long long VR, int *CL_out, int *G_out,
                               int *threads_out, int *maxc_out)
{
    const bool wide_cta = VR > 1024 || (VR > 512 && rows > (size_t)h->R);
    const int ti = VR <= 32 ? 0 : VR <= 64 ? 1 : wide_cta ? 3 : 2;
    const size_t CL = ceil_div(VR, (size_t)kNormThreads[ti]);
    if (CL > SFAR_NORM_CLMAX)
        return SFAR_ERR_UNSUPPORTED;
    int &slot = h->ts_clusters[test][CL][ti];
    if (!slot) {
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)CL);
        cfg.blockDim = dim3((unsigned)kNormThreads[ti]);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int cur = -1, n = 0;
        cudaGetDevice(&cur);
        if (cur != h->dev)
            cudaSetDevice(h->dev);
        const cudaError_t err =
            cudaOccupancyMaxActiveClusters(&n, sfar_kernel_fused_ts(h->dt, h->R > 8, test), &cfg);
        if (cur != h->dev && cur >= 0)
            cudaSetDevice(cur);
        if (err != cudaSuccess) {
            cudaGetLastError();
            return SFAR_ERR_CUDA;
        }
        slot = n > 0 ? n : -1;
    }
    if (slot < h->R)
        return SFAR_ERR_UNSUPPORTED;
    size_t G = (size_t)slot / (size_t)h->R;
    if (G > (size_t)SFAR_KMAX / CL)
        G = (size_t)SFAR_KMAX / CL;
    if (G > ceil_div(rows, (size_t)h->R))
        G = ceil_div(rows, (size_t)h->R);
    *CL_out = (int)CL;
    *G_out = (int)(G < 1 ? 1 : G);
    *threads_out = kNormThreads[ti];
    *maxc_out = slot;
    return SFAR_OK;
}

// The launch plan of a fused call.  8-byte units (one LL line per peer and
// thread, as the plain LL kernel) serve an AllReduce of rows of at most
// 16 KB when every cluster still gets at most one row: they double the
// threads of a row, so a rank gets about half as many clusters, which costs
// more than the shorter receive once a cluster has several rows.  16-byte
// units otherwise, and always for the normalisation alone (no receive).
//
// Path 2, the two-shot fused kernel, serves an AllReduce whose rows (at most
// 32 KB) the one-shot plan would stack several to a cluster: there every
// rank would receive every row from every peer through LL packets, while the
// two-shot owner of a row reads each rank's row once.  Path 1 is the one-shot
// kernel over LL packets; it also takes the shapes whose two-shot grid
// cannot be resident at once.
static sfar_status norm_plan(sfar *h, int allreduce, int test, size_t rows, size_t row_bytes, int *path, int *unit,
                             int *CL, int *G, int *threads, int *vpt, int *batch, int *maxc)
{
    const bool ts_fits = allreduce && row_bytes <= 32768;
    *vpt = 1;
    *batch = 1;
    if (ts_fits && h->fused_path == 2 &&
        ts_geometry(h, test, rows, row_bytes / 16, CL, G, threads, maxc) == SFAR_OK) {
        *path = 2;
        *unit = 16;
        return SFAR_OK;
    }
    *path = 1;
    if (allreduce && row_bytes <= 16384) {
        const sfar_status st =
            norm_geometry(h, allreduce, test, rows, row_bytes / 8, 8, CL, G, threads, vpt, batch, maxc);
        if (st == SFAR_OK && (size_t)*G >= rows) {
            *unit = 8;
            return SFAR_OK;
        }
    }
    *unit = 16;
    const sfar_status st =
        norm_geometry(h, allreduce, test, rows, row_bytes / 16, 16, CL, G, threads, vpt, batch, maxc);
    if (ts_fits && h->fused_path == 0 && (st != SFAR_OK || (size_t)*G < rows)) {
        int tCL = 0, tG = 0, tT = 0, tmax = 0;
        if (ts_geometry(h, test, rows, row_bytes / 16, &tCL, &tG, &tT, &tmax) == SFAR_OK) {
            *path = 2;
            *CL = tCL;
            *G = tG;
            *threads = tT;
            *maxc = tmax;
            *vpt = 1;
            *batch = 1;
            return SFAR_OK;
        }
    }
    return st;
}

static bool ranges_overlap(const void *a, const void *b, size_t bytes)
{
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + bytes && b0 < a0 + bytes;
}

static sfar_status fused_call(sfar *h, const void *const in[], const void *const residual[], const void *weight,
                              void *const out[], void *const residual_out[], size_t rows, size_t hidden, float eps,
                              int allreduce, sfar_stream_t s)
{
    if (!h)
        return SFAR_ERR_INVALID;
    if (allreduce && h->poisoned)
        return SFAR_ERR_POISONED;
    if (rows == 0)
        return SFAR_OK;
    if (!in || !residual || !weight || !out || !residual_out || hidden == 0 || ((uintptr_t)weight & 15u))
        return SFAR_ERR_INVALID;
    const int R = h->R;
    const size_t es = (size_t)h->es;
    if ((hidden * es) % 16 || rows > ((size_t)-1) / 16 / (hidden * es))
        return SFAR_ERR_INVALID;
    const size_t bytes = rows * hidden * es;
    if (allreduce && bytes > h->rb)
        return SFAR_ERR_INVALID;
    // rows of at most 128 KiB (64 KiB for R > 8)
    if (hidden * es > 131072 || (R > 8 && hidden * es > 65536))
        return SFAR_ERR_INVALID;
    for (int r = 0; r < R; ++r)
        if (!in[r] || !residual[r] || !out[r] || !residual_out[r] || ((uintptr_t)in[r] & 15u) ||
            ((uintptr_t)residual[r] & 15u) || ((uintptr_t)out[r] & 15u) || ((uintptr_t)residual_out[r] & 15u))
            return SFAR_ERR_INVALID;
    // writes (out, residual_out) overlap no read (in, residual, weight) and no
    // other write; residual_out[r] == residual[r] (in place) is the exception
    for (int i = 0; i < R; ++i) {
        const void *w[2] = {out[i], residual_out[i]};
        for (int m = 0; m < 2; ++m) {
            if (ranges_overlap(w[m], weight, hidden * es))
                return SFAR_ERR_INVALID;
            for (int j = 0; j < R; ++j) {
                if (ranges_overlap(w[m], in[j], bytes))
                    return SFAR_ERR_INVALID;
                if (ranges_overlap(w[m], residual[j], bytes) && !(m == 1 && j == i && w[m] == residual[j]))
                    return SFAR_ERR_INVALID;
                for (int n = 0; n < 2; ++n) {
                    const void *o = n == 0 ? out[j] : residual_out[j];
                    if ((j != i || n != m) && ranges_overlap(w[m], o, bytes))
                        return SFAR_ERR_INVALID;
                }
            }
        }
    }
    const int test = allreduce && (h->k_strag || h->k_drop || h->k_single) ? 1 : 0;
    int path = 1, unit = 16, CL = 0, G = 0, threads = 0, vpt = 1, batch = 1, maxc = 0;
    const sfar_status gst =
        norm_plan(h, allreduce, test, rows, hidden * es, &path, &unit, &CL, &G, &threads, &vpt, &batch, &maxc);
    if (gst != SFAR_OK)
        return gst;
    const unsigned long long VR = hidden * es / (size_t)unit;
    const int K = G * CL;
    int cur = -1;
    cudaGetDevice(&cur);

    SfarArgs a;
    memset(&a, 0, sizeof a);
    SfarNormArgs na;
    memset(&na, 0, sizeof na);
    for (int r = 0; r < R; ++r) {
        a.in[r] = in[r];
        a.out[r] = out[r];
        na.res[r] = residual[r];
        na.res_out[r] = residual_out[r];
    }
    a.n = rows * hidden;
    a.epoch = h->epoch;
    a.done = h->done;
    a.ctl = h->ctl;
    a.R = R;
    a.K = K;
    a.region = path == 1 ? h->r_ll : nullptr;
    a.slot = path == 1 ? h->s_ll : 0;
    a.fa = path == 2 ? h->fc : nullptr;       // arrival flags [R][KMAX]
    a.fb = path == 2 ? h->fd : nullptr;       // completion flags [R][R][KMAX]
    a.trace = allreduce ? h->trace : nullptr;
    a.trace_calls = allreduce ? h->trace_calls : 0;
    na.weight = weight;
    na.rows = rows;
    na.hidden = hidden;
    na.eps = eps;
    na.G = (int)G;
    na.CL = CL;
    na.vpt = vpt;
    na.B = batch;
    int c = 0;
    while (((size_t)1 << c) < hidden)
        ++c;
    na.F = 53 - c;
    a.overlap = 0;
    // Cooperative mode launches a fused AllReduce grid as a cooperative grid:
    // the device places it whole, so it keeps its programmatic launch and
    // never needs to run solo to be sure that all of its clusters start
    // (measured: no cost at one row, 0.9 us gained at four rows of 8192).
    // It is not the default: Nsight Compute's replay of such a launch ran the
    // grid without its clusters (see wrong_cluster_shape), while the
    // programmatic launch of a plain cluster grid profiles correctly.
    const bool coop = allreduce && h->mode == SFAR_LAUNCH_COOPERATIVE;
    const bool solo = allreduce && !coop && solo_grid(R * G, maxc);
    a.solo = solo ? 1 : 0;
    if (path == 2 || solo) {
        // the two-shot kernel and a solo grid never overtake a call, and the
        // call after them does not overtake them: serial semantics
        h->last_key = -1;
    } else if (allreduce && h->mode == SFAR_LAUNCH_OVERLAP) {
        // the unit -> CTA mapping depends on the cluster shape, the row
        // length and the unit size too, so all of them are part of the
        // overlap key
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        unsigned long long cap = 0;
        if (cudaStreamGetCaptureInfo((cudaStream_t)s, &cs, &cap) != cudaSuccess) {
            cudaGetLastError();
            cs = cudaStreamCaptureStatusNone;
        }
        if (cs != cudaStreamCaptureStatusActive)
            cap = 0;
        const long long key = ((long long)(unit == 8) << 45) | (31ll << 40) | ((long long)CL << 36) |
                              ((long long)K << 27) | ((long long)threads << 16) | (long long)VR;
        a.overlap = (key == h->last_key && s == h->last_stream && cap == h->last_capture) ? 1 : 0;
        h->last_key = key;
        h->last_stream = s;
        h->last_capture = cap;
    }

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(R * K));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.stream = (cudaStream_t)s;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int na_attr = 1;
    if (h->mode != SFAR_LAUNCH_PLAIN && !solo) {
        attr[na_attr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na_attr].val.programmaticStreamSerializationAllowed = 1;
        ++na_attr;
    }
    if (coop) {
        attr[na_attr].id = cudaLaunchAttributeCooperative;
        attr[na_attr].val.cooperative = 1;
        ++na_attr;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na_attr;
    void *args[] = {&a, &na};
    if (cur != h->dev)
        cudaSetDevice(h->dev);
    const void *kern = path == 2 ? sfar_kernel_fused_ts(h->dt, R > 8, test)
                                 : sfar_kernel_fused(h->dt, R > 8, allreduce, test, batch, unit);
    cudaError_t err = cudaLaunchKernelExC(&cfg, kern, args);
    if (cur != h->dev && cur >= 0)
        cudaSetDevice(cur);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return err == cudaErrorCooperativeLaunchTooLarge ? SFAR_ERR_UNSUPPORTED : SFAR_ERR_CUDA;
    }
    return SFAR_OK;
}

sfar_status sfar_test_query_norm_launch(sfar_t *h, size_t rows, size_t hidden, int allreduce, int *ctas_per_rank,
                                        int *cluster_size, int *threads_per_cta)
{
    if (!h || hidden == 0 || rows == 0 || (hidden * (size_t)h->es) % 16)
        return SFAR_ERR_INVALID;
    const size_t row = hidden * (size_t)h->es;
    if (row > 131072 || (h->R > 8 && row > 65536))
        return SFAR_ERR_INVALID;
    int path = 1, unit = 16, CL = 0, G = 0, threads = 0, vpt = 1, batch = 1, maxc = 0;
    const sfar_status st =
        norm_plan(h, allreduce ? 1 : 0, 0, rows, row, &path, &unit, &CL, &G, &threads, &vpt, &batch, &maxc);
    if (st != SFAR_OK)
        return st;
    if (ctas_per_rank)
        *ctas_per_rank = G * CL;
    if (cluster_size)
        *cluster_size = CL;
    if (threads_per_cta)
        *threads_per_cta = threads;
    return SFAR_OK;
}

sfar_status sfar_allreduce_add_rmsnorm(sfar_t *h, const void *const in[], const void *const residual[],
                                       const void *weight, void *const out[], void *const residual_out[],
                                       size_t rows, size_t hidden, float eps, sfar_stream_t s)
{
    return fused_call(h, in, residual, weight, out, residual_out, rows, hidden, eps, 1, s);
}

sfar_status sfar_add_rmsnorm(sfar_t *h, const void *const a[], const void *const residual[], const void *weight,
                             void *const out[], void *const residual_out[], size_t rows, size_t hidden, float eps,
                             sfar_stream_t s)
{
    return fused_call(h, a, residual, weight, out, residual_out, rows, hidden, eps, 0, s);
}

// ------------------------------------------------ row-parallel projection
// The driver's tensor-map encoder, looked up once (no link against the driver library).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            p = nullptr;
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

sfar_status sfar_rowpar_gemv(sfar_t *h, const void *const x[], const void *const w[], void *const y[], size_t k,
                             size_t hidden, size_t prefetch_rows, sfar_stream_t s)
{
    if (!h || !x || !w || !y || h->dt != SFAR_BF16 || k == 0 || hidden == 0 || hidden % 8 || k >= (1ull << 31) ||
        hidden >= (1ull << 31))
        return SFAR_ERR_INVALID;
    const int R = h->R;
    const size_t wbytes = k * hidden * 2, ybytes = hidden * 2, xbytes = k * 2;
    for (int r = 0; r < R; ++r) {
        if (!x[r] || !w[r] || !y[r] || ((uintptr_t)x[r] & 1u) || ((uintptr_t)w[r] & 15u) || ((uintptr_t)y[r] & 15u))
            return SFAR_ERR_INVALID;
    }
    for (int i = 0; i < R; ++i)
        for (int j = 0; j < R; ++j) {
            const uintptr_t y0 = (uintptr_t)y[i], y1 = y0 + ybytes;
            const uintptr_t x0 = (uintptr_t)x[j], x1 = x0 + xbytes, w0 = (uintptr_t)w[j], w1 = w0 + wbytes;
            if ((y0 < x1 && x0 < y1) || (y0 < w1 && w0 < y1))
                return SFAR_ERR_INVALID;
            if (i != j) {
                const uintptr_t z0 = (uintptr_t)y[j], z1 = z0 + ybytes;
                if (y0 < z1 && z0 < y1)
                    return SFAR_ERR_INVALID;
            }
        }
    const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode)
        return SFAR_ERR_UNSUPPORTED;
    SfarGemvArgs g;
    memset(&g, 0, sizeof g);
    const cuuint64_t dims[2] = {(cuuint64_t)hidden, (cuuint64_t)k};
    const cuuint64_t strides[1] = {(cuuint64_t)hidden * 2};
    const cuuint32_t box[2] = {SFAR_GEMV_COLS, SFAR_GEMV_ROWS}, unit[2] = {1, 1};
    for (int r = 0; r < R; ++r) {
        g.x[r] = x[r];
        g.y[r] = y[r];
        if (encode(&g.wmap[r], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(w[r]), dims, strides, box, unit,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return SFAR_ERR_INVALID;
    }
    g.ctl = h->ctl;
    g.k = k;
    g.h = hidden;
    // whole stages of the copy ring, at most the STAGES - 1 that its prologue issues
    const size_t pre = ceil_div(prefetch_rows, SFAR_GEMV_ROWS);
    g.pre = (int)(pre < SFAR_GEMV_STAGES - 1 ? pre : SFAR_GEMV_STAGES - 1);
    g.tiles = (int)ceil_div(hidden, SFAR_GEMV_COLS);

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(R * g.tiles));
    cfg.blockDim = dim3(SFAR_GEMV_THREADS);
    cfg.dynamicSmemBytes = SFAR_GEMV_SMEM;
    cfg.stream = (cudaStream_t)s;
    cudaLaunchAttribute attr[1];
    if (h->mode != SFAR_LAUNCH_PLAIN) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    void *args[] = {&g};
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != h->dev)
        cudaSetDevice(h->dev);
    cudaError_t err = cudaLaunchKernelExC(&cfg, sfar_kernel_gemv(), args);
    if (cur != h->dev && cur >= 0)
        cudaSetDevice(cur);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    return SFAR_OK;
}

sfar_status sfar_status_get(sfar_t *h, sfar_fault *info)
{
    if (!h)
        return SFAR_ERR_INVALID;
    if (cudaMemcpyAsync(h->host_ctl, h->ctl, 32, cudaMemcpyDeviceToHost, h->priv) != cudaSuccess ||
        cudaStreamSynchronize(h->priv) != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    const SfarCtl *c = h->host_ctl;
    const sfar_status code = c->status;
    if (info) {
        info->code = code;
        info->rank = code ? c->f_rank : -1;
        info->cta = code ? c->f_cta : -1;
        info->peer = code ? c->f_peer : -1;
        info->epoch = code ? c->f_epoch : 0;
        info->where = code ? c->f_where : 0;
    }
    if (code != SFAR_OK)
        h->poisoned = true;
    return code;
}

sfar_status sfar_reset(sfar_t *h, sfar_stream_t s)
{
    if (!h)
        return SFAR_ERR_INVALID;
    cudaStream_t st = (cudaStream_t)s;
    if (cudaMemsetAsync(h->ws + h->ctl_bytes, 0, h->ws_bytes - h->ctl_bytes, st) != cudaSuccess ||
        cudaMemsetAsync(h->r_sent, 0xff, h->sent_bytes, st) != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    sfar_status r = launch_knob(h, KNOB_CLEAR_STATUS, 0, nullptr, 0, -1, st);
    if (r == SFAR_OK)
        r = launch_knob(h, KNOB_STRAG, 0, nullptr, 0, -1, st);
    if (r == SFAR_OK)
        r = launch_knob(h, KNOB_DROP, 0, nullptr, 0, -1, st);
    if (r != SFAR_OK)
        return r;
    h->k_strag = false;
    h->k_drop = false;
    h->poisoned = false;
    h->last_key = -1;
    return SFAR_OK;
}

// ------------------------------------------------------------------ test hooks
sfar_status sfar_test_set_straggler(sfar_t *h, const uint32_t *delays_ns, uint32_t len, int rank, int phase,
                                    sfar_stream_t s)
{
    if (!h || (len > 0 && !delays_ns) || rank >= h->R || (phase != 0 && phase != 1))
        return SFAR_ERR_INVALID;
    sfar_status r = launch_knob(h, KNOB_STRAG, 0, delays_ns, len, rank < 0 ? -1 : rank, (cudaStream_t)s, phase);
    if (r == SFAR_OK)
        h->k_strag = len > 0;
    return r;
}

sfar_status sfar_test_drop_rank(sfar_t *h, int rank, sfar_stream_t s)
{
    if (!h || rank >= h->R)
        return SFAR_ERR_INVALID;
    sfar_status r = launch_knob(h, KNOB_DROP, 0, nullptr, 0, rank < 0 ? -1 : rank, (cudaStream_t)s);
    if (r == SFAR_OK)
        h->k_drop = rank >= 0;
    return r;
}

sfar_status sfar_test_set_timeout(sfar_t *h, uint64_t ns, sfar_stream_t s)
{
    if (!h || ns == 0)
        return SFAR_ERR_INVALID;
    return launch_knob(h, KNOB_TIMEOUT, ns, nullptr, 0, -1, (cudaStream_t)s);
}

sfar_status sfar_test_force_single_buffer(sfar_t *h, int on, sfar_stream_t s)
{
    if (!h)
        return SFAR_ERR_INVALID;
    sfar_status r = launch_knob(h, KNOB_SINGLE, on ? 1 : 0, nullptr, 0, -1, (cudaStream_t)s);
    if (r == SFAR_OK)
        h->k_single = on != 0;
    return r;
}

sfar_status sfar_set_launch_mode(sfar_t *h, int mode)
{
    if (!h || (mode != SFAR_LAUNCH_SERIAL && mode != SFAR_LAUNCH_OVERLAP && mode != SFAR_LAUNCH_PLAIN &&
               mode != SFAR_LAUNCH_COOPERATIVE))
        return SFAR_ERR_INVALID;
    h->mode = mode;
    h->last_key = -1;
    return SFAR_OK;
}

sfar_status sfar_test_set_trace(sfar_t *h, uint64_t *trace, uint32_t calls)
{
    if (!h)
        return SFAR_ERR_INVALID;
    if (!trace || calls == 0) {
        h->trace = nullptr;
        h->trace_calls = 0;
    } else {
        h->trace = reinterpret_cast<unsigned long long *>(trace);
        h->trace_calls = calls;
    }
    return SFAR_OK;
}

sfar_status sfar_test_set_geometry(sfar_t *h, int ctas_per_rank, int threads_per_cta)
{
    if (!h || ctas_per_rank < 0 || (threads_per_cta != 0 && thread_index(threads_per_cta) < 0))
        return SFAR_ERR_INVALID;
    h->ctas_override = ctas_per_rank;
    h->threads_override = threads_per_cta;
    return SFAR_OK;
}

sfar_status sfar_test_set_fused_path(sfar_t *h, int path)
{
    if (!h || path < 0 || path > 2)
        return SFAR_ERR_INVALID;
    h->fused_path = path;
    return SFAR_OK;
}

sfar_status sfar_test_query_fused_path(sfar_t *h, size_t rows, size_t hidden, int *path)
{
    if (!h || !path || hidden == 0 || rows == 0 || (hidden * (size_t)h->es) % 16)
        return SFAR_ERR_INVALID;
    const size_t row = hidden * (size_t)h->es;
    if (row > 131072 || (h->R > 8 && row > 65536))
        return SFAR_ERR_INVALID;
    int unit = 16, CL = 0, G = 0, threads = 0, vpt = 1, batch = 1, maxc = 0;
    return norm_plan(h, 1, 0, rows, row, path, &unit, &CL, &G, &threads, &vpt, &batch, &maxc);
}

sfar_status sfar_probe_empty(sfar_stream_t s)
{
    if (cudaLaunchKernel(sfar_kernel_empty(), dim3(1), dim3(32), nullptr, 0, (cudaStream_t)s) != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    return SFAR_OK;
}

sfar_status sfar_probe_pingpong(uint32_t *flags, int trips, int relaxed, int partner, uint64_t *out,
                                sfar_stream_t s)
{
    if (!flags || !out || trips < 1 || partner < 1)
        return SFAR_ERR_INVALID;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    if (partner >= sms)
        return SFAR_ERR_INVALID;
    // > half of an SM's shared memory each: one CTA per SM, all resident at once
    const int smem = 120 * 1024;
    unsigned long long *o = reinterpret_cast<unsigned long long *>(out);
    void *args[] = {&flags, &trips, &relaxed, &partner, &o};
    if (cudaFuncSetAttribute(sfar_kernel_pingpong(), cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
        cudaMemsetAsync(flags, 0, 64 * sizeof(uint32_t), (cudaStream_t)s) != cudaSuccess ||
        cudaLaunchKernel(sfar_kernel_pingpong(), dim3(partner + 1), dim3(32), args, smem, (cudaStream_t)s) !=
            cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    return SFAR_OK;
}

}  // extern "C"
