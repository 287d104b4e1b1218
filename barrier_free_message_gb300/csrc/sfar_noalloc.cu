// sfar_noalloc.cu -- an AllReduce entry point that allocates no memory.
//
// Some callers cannot allocate device memory when they want an AllReduce:
// code running while a stream is being captured into a CUDA graph (cudaMalloc
// is not allowed there), code inside a framework whose caching allocator owns
// all device memory and forbids allocations behind its back, and latency
// paths that cannot pay for cudaMalloc's implicit device synchronisation.
// For them, sfar_allreduce_noalloc runs the one-shot LL kernel of
// sfar_allreduce(..., SFAR_LL, ...) with its working memory (receive region,
// call counters, hand-off flags, status block) taken from one fixed array in
// this file instead of a handle's allocation.
//
// Limits: at most SFAR_NOALLOC_MAX_RANKS ranks and SFAR_NOALLOC_MAX_BYTES
// bytes per rank; the array (about 13 MiB) exists on every GPU that loads the
// library, for the life of the process.  Every call shares it and it keeps
// what the last call left: the call counters must keep counting (never
// cleared between calls), and the receive region is never cleared because
// each call's flags carry a larger epoch than anything left behind.  Calls
// whose kernels overlap on the GPU (concurrent streams) race on the array.
//
// Failures: a bounded device wait that gives up records itself in the
// array's status block, and every later kernel then exits at once.
// sfar_noalloc_status reads that record (and, once it has reported a
// failure, makes later calls return SFAR_ERR_POISONED), or clears it.
#include <cuda_runtime.h>
#include <string.h>

#include <mutex>

#include "sfar.h"
#include "sfar_internal.h"
#include "sfar_test.h"

namespace {

// Layout: the status block, then one block per rank count R = 2..8 holding
// that R's call counters [R] (u64), hand-off flags [R][KMAX] (u32) and LL
// receive region [R][2][R][kSlot].  Calls with different R never share
// counters or slots, so a call with R ranks meets only flags left by earlier
// calls with R ranks, whose epochs are all smaller than its own.
constexpr size_t kCtlBytes = 256;
constexpr size_t kSlot = 2 * (size_t)SFAR_NOALLOC_MAX_BYTES;            // LL: 2 wire bytes per byte
constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t counters_bytes(int R) { return align256((size_t)R * 8); }
constexpr size_t done_bytes(int R) { return align256((size_t)R * SFAR_KMAX * 4); }
constexpr size_t block_bytes(int R)
{
    return counters_bytes(R) + done_bytes(R) + (size_t)R * 2 * R * kSlot;
}
constexpr size_t block_offset(int R)      // offset of rank count R's block
{
    size_t off = kCtlBytes;
    for (int q = 2; q < R; ++q)
        off += block_bytes(q);
    return off;
}
constexpr size_t kScratchBytes = block_offset(SFAR_NOALLOC_MAX_RANKS + 1);
static_assert(sizeof(SfarCtl) <= kCtlBytes, "status block does not fit");
static_assert(kScratchBytes < (16u << 20), "the array must stay modest");

constexpr int kThreads = 64;
constexpr int kMaxDevices = 64;

}  // namespace

// The working memory of sfar_allreduce_noalloc (see the header comment).
static __device__ __align__(256) unsigned char g_sfar_noalloc_scratch[kScratchBytes];

// Zero the array and write the status block's defaults (device code may name
// the array directly).
__global__ void k_noalloc_init(unsigned long long timeout_ns)
{
    const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const size_t nthreads = (size_t)gridDim.x * blockDim.x;
    uint4 *p = reinterpret_cast<uint4 *>(g_sfar_noalloc_scratch + kCtlBytes);
    const size_t nvec = (kScratchBytes - kCtlBytes) / 16;
    for (size_t i = tid; i < nvec; i += nthreads)
        p[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        SfarCtl *c = reinterpret_cast<SfarCtl *>(g_sfar_noalloc_scratch);
        memset(c, 0, sizeof(SfarCtl));
        c->timeout_ns = timeout_ns;
        c->f_rank = c->f_cta = c->f_peer = -1;
        c->strag_rank = -1;
        c->drop_rank = -1;
    }
}

namespace {

std::mutex g_mu;
unsigned char *g_ptr[kMaxDevices];     // device address of the array, per device
bool g_ready[kMaxDevices];
bool g_poisoned[kMaxDevices];          // a device-side failure was reported and not cleared

// The status block's first 32 bytes: the code and the fault record.
struct FaultRecord {
    int status, f_rank, f_cta, f_peer;
    uint32_t f_epoch;
    int f_where;
    int pad[2];
};
static_assert(sizeof(FaultRecord) == 32, "status block prefix");

// Once per device, with that device current: find the array's device address
// (in host code its name is only a stand-in), check that the grid of the
// largest call can be resident at once, and clear the array.  Synchronises
// the stream, so the first call must not be made under stream capture.
sfar_status setup(int dev, cudaStream_t s, unsigned char **out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_ready[dev]) {
        *out = g_ptr[dev];
        return SFAR_OK;
    }
    int major = 0, minor = 0, sms = 0, nb = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    if (major != 10 || minor != 3)
        return SFAR_ERR_UNSUPPORTED;
    for (int dt = 0; dt < 2; ++dt) {
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, sfar_kernel_ll(dt, 0, 0), kThreads, 0) !=
            cudaSuccess) {
            cudaGetLastError();
            return SFAR_ERR_CUDA;
        }
        const int most = SFAR_NOALLOC_MAX_RANKS * (SFAR_NOALLOC_MAX_BYTES / SFAR_LL_UNIT_NARROW / kThreads);
        if (nb * sms < most)
            return SFAR_ERR_UNSUPPORTED;
    }
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_sfar_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    k_noalloc_init<<<sms, 256, 0, s>>>(1000000000ull);
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    g_ptr[dev] = static_cast<unsigned char *>(ptr);
    g_ready[dev] = true;
    *out = g_ptr[dev];
    return SFAR_OK;
}

}  // namespace

extern "C" sfar_status sfar_allreduce_noalloc(const void *const in[], void *const out[], int R, size_t n,
                                              sfar_dtype dt, sfar_stream_t s)
{
    if (R < 2 || R > SFAR_NOALLOC_MAX_RANKS || (dt != SFAR_BF16 && dt != SFAR_FP32))
        return SFAR_ERR_INVALID;
    if (n == 0)
        return SFAR_OK;
    const size_t es = dt == SFAR_BF16 ? 2 : 4;
    if (!in || !out || n > SFAR_NOALLOC_MAX_BYTES / es)
        return SFAR_ERR_INVALID;
    const size_t bytes = n * es;
    for (int r = 0; r < R; ++r)
        if (!in[r] || !out[r] || ((uintptr_t)in[r] & 15u) || ((uintptr_t)out[r] & 15u))
            return SFAR_ERR_INVALID;
    for (int i = 0; i < R; ++i) {
        const uintptr_t o0 = (uintptr_t)out[i], o1 = o0 + bytes;
        for (int j = 0; j < R; ++j) {
            const uintptr_t a0 = (uintptr_t)in[j], a1 = a0 + bytes;
            if (o0 < a1 && a0 < o1)
                return SFAR_ERR_INVALID;
            const uintptr_t b0 = (uintptr_t)out[j], b1 = b0 + bytes;
            if (j != i && o0 < b1 && b0 < o1)
                return SFAR_ERR_INVALID;
        }
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    unsigned char *base = nullptr;
    const sfar_status st = setup(dev, (cudaStream_t)s, &base);
    if (st != SFAR_OK)
        return st;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_poisoned[dev])
            return SFAR_ERR_POISONED;
    }

    SfarArgs a;
    memset(&a, 0, sizeof a);
    for (int r = 0; r < R; ++r) {
        a.in[r] = in[r];
        a.out[r] = out[r];
    }
    const size_t units = (bytes + SFAR_LL_UNIT_NARROW - 1) / SFAR_LL_UNIT_NARROW;     // the LL kernel's units
    const int K = (int)((units + kThreads - 1) / kThreads);
    unsigned char *blk = base + block_offset(R);
    a.n = n;
    a.slot = kSlot;
    a.epoch = reinterpret_cast<unsigned long long *>(blk);
    a.done = reinterpret_cast<uint32_t *>(blk + counters_bytes(R));
    a.region = blk + counters_bytes(R) + done_bytes(R);
    a.ctl = reinterpret_cast<SfarCtl *>(base);
    a.R = R;
    a.K = K;
    a.overlap = 0;

    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(R * K));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = (cudaStream_t)s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&a};
    if (cudaLaunchKernelExC(&cfg, sfar_kernel_ll((int)dt, 0, 0), args) != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    return SFAR_OK;
}

namespace {

sfar_status current_device(int *dev)
{
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kMaxDevices) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    return SFAR_OK;
}

sfar_status write_record(unsigned char *base, const FaultRecord &rec)
{
    if (cudaMemcpy(base, &rec, sizeof rec, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    return SFAR_OK;
}

}  // namespace

extern "C" sfar_status sfar_noalloc_status(sfar_fault *info, int clear)
{
    int dev = 0;
    sfar_status st = current_device(&dev);
    if (st != SFAR_OK)
        return st;
    unsigned char *base = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (g_ready[dev])
            base = g_ptr[dev];
    }
    FaultRecord rec;
    memset(&rec, 0, sizeof rec);
    if (base && cudaMemcpy(&rec, base, sizeof rec, cudaMemcpyDeviceToHost) != cudaSuccess) {
        cudaGetLastError();
        return SFAR_ERR_CUDA;
    }
    const sfar_status code = rec.status;
    if (info) {
        info->code = code;
        info->rank = code ? rec.f_rank : -1;
        info->cta = code ? rec.f_cta : -1;
        info->peer = code ? rec.f_peer : -1;
        info->epoch = code ? rec.f_epoch : 0;
        info->where = code ? rec.f_where : 0;
    }
    if (clear && base) {
        FaultRecord zero;
        memset(&zero, 0, sizeof zero);
        zero.f_rank = zero.f_cta = zero.f_peer = -1;
        st = write_record(base, zero);
        if (st != SFAR_OK)
            return st;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    g_poisoned[dev] = clear ? false : (g_poisoned[dev] || code != SFAR_OK);
    return code;
}

extern "C" sfar_status sfar_test_noalloc_record_failure(int rank, int peer, int where)
{
    int dev = 0;
    sfar_status st = current_device(&dev);
    if (st != SFAR_OK)
        return st;
    unsigned char *base = nullptr;
    st = setup(dev, nullptr, &base);
    if (st != SFAR_OK)
        return st;
    FaultRecord rec;
    memset(&rec, 0, sizeof rec);
    rec.status = SFAR_ERR_TIMEOUT;
    rec.f_rank = rank;
    rec.f_cta = 0;
    rec.f_peer = peer;
    rec.f_where = where;
    return write_record(base, rec);
}
