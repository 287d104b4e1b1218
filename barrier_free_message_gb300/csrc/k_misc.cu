// k_misc.cu -- knob writes and the latency-floor probes.
//
// The floor a one-shot AllReduce of a few KB cannot beat on one GPU is one
// kernel launch plus one flag hand-off through L2 between two SMs; it stands
// in for the pages' speed-of-light bound ("Every Microsecond Counts"
// (page 1), section "Tensor parallelism and AllReduce": the kernel came
// within 7% of the hardware limit).  The probes measure the two parts.
#include "sfar_prims.cuh"

__global__ void k_set_knob(const SfarKnobArgs k)
{
    SfarCtl *c = k.ctl;
    switch (k.which) {
    case KNOB_TIMEOUT:
        c->timeout_ns = k.value;
        break;
    case KNOB_STRAG:
        c->strag_delays = k.ptr;
        c->strag_len = k.len;
        c->strag_rank = k.rank;
        c->strag_phase = k.phase;
        c->strag_base = (uint32_t)(k.epoch0[0] / SFAR_KMAX);
        break;
    case KNOB_DROP:
        c->drop_rank = k.rank;
        break;
    case KNOB_SINGLE:
        c->single_buffer = (int)k.value;
        break;
    case KNOB_CLEAR_STATUS:
        c->status = 0;
        c->f_rank = c->f_cta = c->f_peer = -1;
        c->f_epoch = 0;
        c->f_where = 0;
        break;
    default:
        break;
    }
}

__global__ void k_empty() {}

// Two CTAs (forced onto different SMs by their shared-memory size) pass a
// token back and forth through two flags 128 bytes apart.  relaxed = 0:
// st.release / ld.acquire at GPU scope (a flag that publishes data); 1:
// relaxed stores and loads (the cost of the hand-off alone, as in LL).
__device__ __forceinline__ void pp_store(uint32_t *p, uint32_t v, int relaxed)
{
    if (relaxed)
        st_relaxed_u32(p, v);
    else
        st_release_u32(p, v);
}
__device__ __forceinline__ uint32_t pp_load(const uint32_t *p, int relaxed)
{
    return relaxed ? ld_relaxed_u32(p) : ld_acquire_u32(p);
}

// The grid has one CTA per SM (shared-memory size); CTA 0 and CTA `partner`
// play, the others leave at once.  out[1], out[2] get the two SM ids.
__global__ void k_pingpong(uint32_t *flags, int trips, int relaxed, int partner, unsigned long long *out)
{
    extern __shared__ uint8_t pad[];
    if (threadIdx.x != 0 || (blockIdx.x != 0 && (int)blockIdx.x != partner))
        return;
    pad[0] = 0;
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    out[blockIdx.x == 0 ? 1 : 2] = smid;
    unsigned long long *ns_out = out;
    uint32_t *ping = flags, *pong = flags + 32;
    const unsigned long long limit = 1000000000ull;
    const unsigned long long start = globaltimer();
    bool ok = true;
    if (blockIdx.x == 0) {
        for (int i = 1; i <= trips && ok; ++i) {
            pp_store(ping, (uint32_t)i, relaxed);
            uint32_t it = 0;
            while (pp_load(pong, relaxed) != (uint32_t)i)
                if ((++it & 255u) == 0 && globaltimer() - start > limit) {
                    ok = false;
                    break;
                }
        }
        *ns_out = ok ? globaltimer() - start : ~0ull;
        if (!ok)
            st_release_u32(ping, 0xffffffffu);
    } else {
        for (int i = 1; i <= trips && ok; ++i) {
            uint32_t it = 0, v;
            while ((v = pp_load(ping, relaxed)) != (uint32_t)i) {
                if (v == 0xffffffffu || ((++it & 255u) == 0 && globaltimer() - start > limit)) {
                    ok = false;
                    break;
                }
            }
            if (ok)
                pp_store(pong, (uint32_t)i, relaxed);
        }
    }
}

const void *sfar_kernel_set_knob() { return (const void *)k_set_knob; }
const void *sfar_kernel_empty() { return (const void *)k_empty; }
const void *sfar_kernel_pingpong() { return (const void *)k_pingpong; }
