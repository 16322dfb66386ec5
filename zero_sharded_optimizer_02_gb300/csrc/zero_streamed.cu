// Bucket-ready shard step: the optimizer starts on a bucket as soon as its
// reduced gradients have landed (sm_103a).
//
// "ZeRO: Memory Optimizations Toward Training Trillion Parameter Models",
// section "ZeRO-DP", Stage 2: gradients are reduce-scattered bucket by bucket
// during the backward pass.  Here the producer of a bucket -- in one GPU's
// emulation, a copy stream landing the bucket's Nd contribution slices --
// writes the bucket's ready word after its data.  The consumer is the fused
// step itself, launched group of buckets by group on one stream, each
// group's launches behind a one-thread kernel that waits for the group's
// ready words.  The step kernels therefore run at their full rate on data that no
// longer changes, and only the waits run while a bucket is in flight.
//
// Every wait is bounded: the waiting thread polls the word with an acquire
// load, sleeping between polls (64 ns, doubling up to about 1 us), for at
// most timeout_ns of %globaltimer time and an iteration cap.  On expiry it
// records ZERO_ERR_TIMEOUT in the status word; every later wait and step
// launch of the call reads the status word first and does nothing, so no
// element of a bucket that was not seen ready is touched, and the context
// stays usable.  The wait never depends on another kernel: only on a word
// written by a copy engine or the host.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include "zero_device.cuh"

namespace zero {
namespace {

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Longest sleep between two polls of a ready word (one thread polls).
#ifndef ZERO_POLL_MAX_NS
#define ZERO_POLL_MAX_NS 1024
#endif

// Bounded wait for *word >= epoch (by wrap-around comparison).  The sleep
// between polls doubles from 64 ns up to ZERO_POLL_MAX_NS.
__device__ bool wait_ready(const uint32_t* word, uint32_t epoch, uint64_t timeout_ns)
{
    const uint64_t t0 = global_ns();
    const uint64_t max_polls = timeout_ns / 64 + 16;   // backstop to the time limit
    unsigned sleep_ns = 64;
    for (uint64_t i = 0; i < max_polls; ++i) {
        if ((int32_t)(ld_acquire(word) - epoch) >= 0)
            return true;
        if (global_ns() - t0 > timeout_ns)
            return false;
        __nanosleep(sleep_ns);
        if (sleep_ns < ZERO_POLL_MAX_NS)
            sleep_ns *= 2;
    }
    return (int32_t)(ld_acquire(word) - epoch) >= 0;
}

// One launch group's wait: a single thread polls the ready words of `count`
// consecutive buckets in order (each wait bounded).  If an earlier wait of
// the call ran out (status nonzero), it does not wait again.
//
// Launched as a programmatic dependent launch, it starts while the previous
// group's step kernel is still running: it lets the next group's launch be
// scheduled at once, polls, and only then waits (griddepcontrol.wait) for
// its predecessor in the stream to complete.  It therefore never completes
// before that kernel, so every later kernel that waits for its own
// predecessor also waits for all earlier ones; the next group's step kernel
// starts as the previous one drains, as between two launch windows.  On a
// plain launch both instructions are no-ops and the kernel runs after its
// predecessor, as before.
__global__ void k_wait_ready(const uint32_t* words, uint64_t count, uint32_t epoch,
                             uint64_t timeout_ns, uint32_t* status)
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (ld_acquire(status) == 0) {
        for (uint64_t i = 0; i < count; ++i)
            if (!wait_ready(words + i, epoch, timeout_ns)) {
                atomicCAS(status, 0u, (uint32_t)ZERO_ERR_TIMEOUT);
                break;
            }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// k_wait_ready on `stream`, as a programmatic dependent launch unless
// ZERO_PDL is "0".
cudaError_t launch_wait(cudaStream_t stream, const uint32_t* words, uint64_t count,
                        uint32_t epoch, uint64_t timeout_ns, uint32_t* status)
{
    if (!pdl_launches()) {
        k_wait_ready<<<1, 1, 0, stream>>>(words, count, epoch, timeout_ns, status);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_wait_ready, words, count, epoch, timeout_ns, status);
}

bool is_aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// ceil(n / bucket) for any bucket >= 1 (no overflow for a bucket near 2^64).
uint64_t buckets_of(uint64_t n, uint64_t bucket) { return n / bucket + (n % bucket != 0); }

}  // namespace
}  // namespace zero

using namespace zero;

extern "C" zero_status_t zero_step_shard_streamed(
    const zero_grads_t* g, const zero_layout_t* L, const zero_state_t* in,
    const zero_state_t* out, void* gathered, uint64_t gathered_offset_elems,
    uint64_t bucket_elems, double loss_scale, const zero_adamw_t* h, const uint32_t* d_ready,
    uint32_t epoch, uint64_t timeout_ns, uint32_t* d_nonfinite, uint32_t* d_status,
    void* stream)
{
    zero_status_t rs = check_step_args(g, L, in, out, gathered, gathered_offset_elems,
                                       bucket_elems, loss_scale, h, d_nonfinite);
    if (rs != ZERO_OK)
        return rs;
    if (!d_ready || !d_status)
        return ZERO_ERR_INVALID_ARG;
    if (timeout_ns == 0 || timeout_ns > ZERO_MAX_WAIT_NS)
        return ZERO_ERR_INVALID_ARG;   // every device wait must stay bounded
    if (!is_aligned(d_ready, 4) || !is_aligned(d_status, 4))
        return ZERO_ERR_ALIGNMENT;
    const uint64_t n = L->length;
    if (n == 0)
        return ZERO_OK;
    bool host_rows = false;
    zero_grads_t gr;   // the rows at the address the device reads them
    rs = resolve_grads(g, &gr, &host_rows);
    if (rs != ZERO_OK)
        return rs;
    void* gdev = nullptr;   // the gathered buffer at the address the device writes it
    rs = resolve_ptr(gathered, &gdev);
    if (rs != ZERO_OK)
        return rs;
    rs = require_device_state(in, out, d_nonfinite);
    if (rs != ZERO_OK)
        return rs;
    const void* words[2] = {d_ready, d_status};
    rs = require_device(words, 2);
    if (rs != ZERO_OK)
        return rs;
    // every kernel this call launches is loaded before its first wait starts
    preload_fused(g->dtype, host_rows);
    const StepScalars k = make_scalars(h, g->nd, loss_scale);
    const uint16_t* rows = static_cast<const uint16_t*>(gr.base) + g->offset;
    uint16_t* gath = static_cast<uint16_t*>(gdev) + gathered_offset_elems;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Consecutive buckets form launch groups: as many groups as the shard's
    // step traffic holds ZERO_STREAM_GROUP_BYTES (the environment variable of
    // that name, read at each call, overrides it; 0: one group a bucket), the
    // buckets dealt as evenly as possible, so that each group's launches
    // outweigh their fixed cost.  A group starts once all its buckets landed.
    uint64_t group_bytes = ZERO_STREAM_GROUP_BYTES;
    if (const char* e = getenv("ZERO_STREAM_GROUP_BYTES")) {
        char* end = nullptr;
        const unsigned long long v = strtoull(e, &end, 10);
        if (end != e && *end == '\0')
            group_bytes = v;
    }
    const uint64_t nb = buckets_of(n, bucket_elems);
    const uint64_t traffic = n * (2ull * g->nd + 26);
    uint64_t ngroups = group_bytes ? traffic / group_bytes : nb;
    ngroups = ngroups < 1 ? 1 : (ngroups > nb ? nb : ngroups);
    const uint64_t base = nb / ngroups, extra = nb % ngroups;   // buckets per group
    for (uint64_t grp = 0, b = 0; grp < ngroups; ++grp) {
        const uint64_t g0 = b * bucket_elems;
        const uint64_t b_end = b + base + (grp < extra ? 1 : 0);
        const uint64_t glen = (b_end * bucket_elems < n ? b_end * bucket_elems : n) - g0;
        if (launch_wait(st, d_ready + b, b_end - b, epoch, timeout_ns, d_status) != cudaSuccess)
            return ZERO_ERR_CUDA;
        const zero_status_t ls = launch_fused_range(rows, g, in, out, gath, g0, glen, k,
                                                     host_rows, d_nonfinite, d_status, stream);
        if (ls != ZERO_OK)
            return ls;
        b = b_end;
    }
    return ZERO_OK;
}

extern "C" zero_status_t zero_feed_buckets(const void* host, uint64_t host_row_stride,
                                           const zero_grads_t* g, uint64_t n,
                                           uint64_t bucket_elems, uint32_t* d_ready,
                                           const uint32_t* h_epoch, void* copy_stream)
{
    if (!host || !g || !g->base || g->nd == 0 || g->nd > ZERO_MAX_ND || !d_ready || !h_epoch ||
        bucket_elems == 0)
        return ZERO_ERR_INVALID_ARG;
    if (host_row_stride < n || g->row_stride < g->offset + n ||
        host_row_stride > (1ull << 60) / 2 || g->row_stride > (1ull << 60) / 2)
        return ZERO_ERR_INVALID_ARG;
    if (!is_aligned(host, 2) || !is_aligned(g->base, 2) || !is_aligned(d_ready, 4) ||
        !is_aligned(h_epoch, 4))
        return ZERO_ERR_ALIGNMENT;
    cudaStream_t st = static_cast<cudaStream_t>(copy_stream);
    const char* src = static_cast<const char*>(host);
    char* dst = const_cast<char*>(static_cast<const char*>(g->base)) + 2 * g->offset;
    const uint64_t nb = buckets_of(n, bucket_elems);
    for (uint64_t b = 0; b < nb; ++b) {
        const uint64_t b0 = b * bucket_elems;
        const uint64_t len = n - b0 < bucket_elems ? n - b0 : bucket_elems;
        // the bucket's slice of every contributor row, then its ready word
        if (cudaMemcpy2DAsync(dst + 2 * b0, 2 * g->row_stride, src + 2 * b0,
                              2 * host_row_stride, 2 * len, g->nd, cudaMemcpyHostToDevice,
                              st) != cudaSuccess ||
            cudaMemcpyAsync(d_ready + b, h_epoch, sizeof(uint32_t), cudaMemcpyHostToDevice,
                            st) != cudaSuccess)
            return ZERO_ERR_CUDA;
    }
    return ZERO_OK;
}
