// Bucket-ready shard step: the optimizer starts on a bucket as soon as its
// reduced gradients have landed (sm_103a).
//
// "ZeRO: Memory Optimizations Toward Training Trillion Parameter Models",
// section "ZeRO-DP", Stage 2: gradients are reduce-scattered bucket by bucket
// during the backward pass.  Here the producer of a bucket -- in one GPU's
// emulation, a copy stream landing the bucket's Nd contribution slices --
// writes the bucket's ready word after its data.  One persistent kernel walks
// the shard's 8-element vectors grid-stride, each thread in increasing order,
// and processes a vector once every bucket it touches is known to be ready.
// There is no barrier per bucket, so a thread never idles at a bucket's end
// while others finish it: when the buckets are already resident the kernel
// is one even pass over the shard.
//
// Readiness is cached per CTA in shared memory ("buckets [0, upto) are
// ready").  A thread that needs a later bucket elects itself poller (one per
// CTA at a time) and polls the ready words in bucket order with acquire loads,
// sleeping between polls (64 ns, doubling up to about 16 us), for at most
// timeout_ns of %globaltimer time a bucket and an iteration cap; the other
// threads sleep on the shared cache, bounded the same way while it makes no
// progress.  On expiry ZERO_ERR_TIMEOUT is recorded in the status word, the
// CTA's threads stop before touching a bucket that is not ready, and the
// context stays usable.  The kernel never waits on another kernel: only on a
// word written by a copy engine or the host.
#include <cuda_runtime.h>
#include <stdint.h>

#include "zero_device.cuh"

namespace zero {
namespace {

constexpr int kStreamThreads = 256;
constexpr int kStreamCtasPerSm = 2;

// Gradient loads of this kernel read data that arrives while it runs, so they
// go through L2 (.cg) instead of the non-coherent path.
__device__ __forceinline__ uint4 ld_grad16_cg(const uint16_t* p)
{
    return __ldcg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ uint16_t ld_grad2_cg(const uint16_t* p)
{
    return __ldcg(reinterpret_cast<const unsigned short*>(p));
}

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Longest sleep between two polls of a ready word.  Every CTA polls the same
// word, so frequent polls pile onto one L2 slice and slow the copy engine's
// writes of the bucket itself.  A bucket takes milliseconds to land over the
// host link; polling every ~16 us delays only the last bucket, by as much.
#ifndef ZERO_POLL_MAX_NS
#define ZERO_POLL_MAX_NS 16384
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

template <int DT>
__device__ __forceinline__ void fold8_cg(const uint16_t* gp, uint64_t row_stride, uint32_t nd,
                                         float (&acc)[8])
{
    set8<DT>(acc, ld_grad16_cg(gp));
    for (uint32_t j0 = 1; j0 < nd; j0 += kRankUnroll) {
        uint4 w[kRankUnroll];
#pragma unroll
        for (int u = 0; u < kRankUnroll; ++u)
            if (j0 + u < nd)
                w[u] = ld_grad16_cg(gp + (uint64_t)(j0 + u) * row_stride);
#pragma unroll
        for (int u = 0; u < kRankUnroll; ++u)
            if (j0 + u < nd)
                add8<DT>(acc, w[u]);
    }
}

struct StreamArgs {
    FusedArgs a;           // one launch window: pointers at its first element, a.sp its split
    uint64_t e0;           // shard element of the window's element 0
    uint64_t bucket;       // bucket size (elements)
    const uint32_t* ready; // ready word of each bucket of the shard
    uint32_t epoch;
    uint64_t timeout_ns;
    uint32_t* status;      // ZERO_ERR_TIMEOUT is recorded here on expiry
};

__device__ __forceinline__ uint32_t ld_acquire_cta(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.cta.shared.u32 %0, [%1];"
                 : "=r"(v)
                 : "r"(smem_u32(p))
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_release_cta(uint32_t* p, uint32_t v)
{
    asm volatile("st.release.cta.shared.u32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// A CTA's shared readiness cache.
struct ReadyCache {
    uint32_t upto;     // buckets [0, upto) are ready
    uint32_t poller;   // 1 while a thread of the CTA polls the ready words
    uint32_t abort;    // 1 once a wait ran out
};

// Waits until buckets [0, need] are known ready.  False if a wait ran out
// (here or in another thread of the CTA); the status word then holds
// ZERO_ERR_TIMEOUT.
__device__ bool wait_buckets(ReadyCache& rc, const StreamArgs& s, uint32_t need)
{
    uint64_t t0 = global_ns();
    uint32_t seen = ld_acquire_cta(&rc.upto);
    unsigned sleep_ns = 32;
    for (uint64_t i = 0; i < (1ull << 40); ++i) {
        const uint32_t u = ld_acquire_cta(&rc.upto);
        if (u > need)
            return true;
        if (ld_acquire_cta(&rc.abort))
            return false;
        if (u != seen) {                       // progress: restart the clock
            seen = u;
            t0 = global_ns();
        }
        if (atomicCAS(&rc.poller, 0u, 1u) == 0u) {
            // the elected poller: ready words in bucket order, one wait each
            uint32_t v = ld_acquire_cta(&rc.upto);
            bool ok = true;
            while (v <= need) {
                if (!wait_ready(s.ready + v, s.epoch, s.timeout_ns)) {
                    ok = false;
                    break;
                }
                st_release_cta(&rc.upto, ++v);
            }
            if (!ok) {
                atomicCAS(s.status, 0u, (uint32_t)ZERO_ERR_TIMEOUT);
                st_release_cta(&rc.abort, 1u);
            }
            atomicExch(&rc.poller, 0u);
            if (!ok)
                return false;
            continue;
        }
        // another thread polls: bounded by the poller's own limit plus margin
        if (global_ns() - t0 > 2 * s.timeout_ns + 1000000) {
            atomicCAS(s.status, 0u, (uint32_t)ZERO_ERR_TIMEOUT);
            st_release_cta(&rc.abort, 1u);
            return false;
        }
        __nanosleep(sleep_ns);
        if (sleep_ns < 1024)
            sleep_ns *= 2;
    }
    atomicCAS(s.status, 0u, (uint32_t)ZERO_ERR_TIMEOUT);
    st_release_cta(&rc.abort, 1u);
    return false;
}

// Scalar element e of the shard (head or tail): fold with .cg loads, AdamW,
// cast.  Returns "sum nonfinite".
template <int DT>
__device__ __forceinline__ bool streamed_scalar(const FusedArgs& a, uint64_t e)
{
    float g = widen1<DT>(ld_grad2_cg(a.g + e));
    for (uint32_t j = 1; j < a.nd; ++j)
        g = __fadd_rn(g, widen1<DT>(ld_grad2_cg(a.g + e + (uint64_t)j * a.row_stride)));
    float p = a.p_in[e], m = a.m_in[e], v = a.v_in[e];
    adamw1(a.k, __fmul_rn(g, a.k.inv), p, m, v);
    a.p_out[e] = p;
    a.m_out[e] = m;
    a.v_out[e] = v;
    a.gath[e] = narrow1<DT>(p);
    return nonfinite(g);
}

template <int DT, int W, bool V8>
__global__ void __launch_bounds__(kStreamThreads, kStreamCtasPerSm) k_step_streamed(const StreamArgs s)
{
    __shared__ ReadyCache rc;
    const uint32_t first_bucket = (uint32_t)(s.e0 / s.bucket);
    if (threadIdx.x == 0) {
        rc.upto = first_bucket;          // earlier buckets belong to earlier windows
        rc.poller = 0;
        rc.abort = 0;
    }
    __syncthreads();
    bool bad = false;
    const uint64_t tid = (uint64_t)blockIdx.x * kStreamThreads + threadIdx.x;
    const uint64_t nthr = (uint64_t)gridDim.x * kStreamThreads;
    const FusedArgs& a = s.a;            // the window; a.sp splits it
    // buckets below `known` are seen ready by this thread: window elements
    // below `ready_end` (kept so that the common case costs one compare)
    uint32_t known = first_bucket;
    uint64_t ready_end = 0;
    auto ready_for = [&](uint64_t last_elem) {
        if (last_elem < ready_end)
            return true;
        const uint32_t need = (uint32_t)((s.e0 + last_elem) / s.bucket);
        if (need >= known) {
            if (!wait_buckets(rc, s, need))
                return false;
            known = need + 1;
        }
        ready_end = (uint64_t)known * s.bucket - s.e0;
        return true;
    };
    bool ok = true;
    // head scalars, then the vectors in order, then the tail
    const uint64_t nscalar = a.sp.nscalar();
    const bool head_scalar = tid < nscalar && tid < a.sp.head;
    if (head_scalar) {
        ok = ready_for(tid);
        if (ok)
            bad |= streamed_scalar<DT>(a, tid);
    }
    for (uint64_t q = tid; ok && q < a.sp.nvec; q += nthr) {
        const uint64_t e = a.sp.head + 8 * q;
        if (!(ok = ready_for(e + 7)))
            break;
        float acc[8];
        fold8_cg<DT>(a.g + e, a.row_stride, a.nd, acc);
        bad |= fused_epilogue<DT, W, V8>(a, e, acc);
    }
    if (ok && tid < nscalar && !head_scalar) {
        const uint64_t e = a.sp.scalar_elem(tid);
        if (ready_for(e))
            bad |= streamed_scalar<DT>(a, e);
    }
    flag_if_any(bad, s.a.flag);
}

int sms_streamed()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        sms = 1;
    return sms;
}

bool is_aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

bool overlap(const void* a, const void* b, uint64_t bytes)
{
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + bytes && y < x + bytes;
}

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
    if (!g || !L || !in || !out || !gathered || !h || !d_ready || !d_nonfinite || !d_status ||
        bucket_elems == 0 || !(loss_scale > 0.0 && loss_scale <= 1.0e300) || !adamw_valid(h))
        return ZERO_ERR_INVALID_ARG;
    if (timeout_ns == 0 || timeout_ns > ZERO_MAX_WAIT_NS)
        return ZERO_ERR_INVALID_ARG;   // every device wait must stay bounded
    if (!g->base || g->nd == 0 || (g->dtype != ZERO_F16 && g->dtype != ZERO_BF16) ||
        L->length > L->shard_elems)
        return ZERO_ERR_INVALID_ARG;
    if (!is_aligned(g->base, 16) || (g->row_stride & 7) || (g->offset & 7) ||
        !is_aligned(gathered, 2) || !is_aligned(d_ready, 4) || !is_aligned(d_nonfinite, 4) ||
        !is_aligned(d_status, 4))
        return ZERO_ERR_ALIGNMENT;
    const float* ins[3] = {in->master, in->m, in->v};
    float* outs[3] = {out->master, out->m, out->v};
    const uint64_t n = L->length;
    const uint64_t lim = 1ull << 61;   // element indices stay far from overflow
    if (n > lim || g->offset > lim - n ||
        (g->nd > 1 && g->row_stride > (lim - g->offset - n) / (g->nd - 1)))
        return ZERO_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i) {
        if (!ins[i] || !outs[i])
            return ZERO_ERR_INVALID_ARG;
        if (!is_aligned(ins[i], 16) || !is_aligned(outs[i], 16))
            return ZERO_ERR_ALIGNMENT;
        for (int j = 0; j < 3; ++j)
            if (!(i == j && outs[i] == ins[j]) && overlap(outs[i], ins[j], n * 4))
                return ZERO_ERR_INVALID_ARG;
    }
    if (n == 0)
        return ZERO_OK;
    zero_grads_t gr;   // the rows at the address the device reads them
    const zero_status_t rs = resolve_grads(g, &gr);
    if (rs != ZERO_OK)
        return rs;
    StreamArgs base;
    base.a.g = static_cast<const uint16_t*>(gr.base) + g->offset;
    base.a.row_stride = g->row_stride;
    base.a.nd = g->nd;
    base.a.p_in = in->master;
    base.a.m_in = in->m;
    base.a.v_in = in->v;
    base.a.p_out = out->master;
    base.a.m_out = out->m;
    base.a.v_out = out->v;
    base.a.gath = static_cast<uint16_t*>(gathered) + gathered_offset_elems;
    base.a.k = make_scalars(h, g->nd, loss_scale);
    base.a.flag = d_nonfinite;
    base.bucket = bucket_elems;
    base.ready = d_ready;
    base.epoch = epoch;
    base.timeout_ns = timeout_ns;
    base.status = d_status;
    // Windows start at multiples of 8 shard elements (offset is one), so
    // every vector of every window has the gathered phase of element 0 and
    // one store width fits all.
    const uintptr_t a0 = (uintptr_t)base.a.gath;
    const int width = (a0 & 15) == 0 ? 16 : (a0 & 7) == 0 ? 8 : (a0 & 3) == 0 ? 4 : 2;
    const float* const sp[6] = {in->master, in->m, in->v, out->master, out->m, out->v};
    const bool v8 = state_v8_ok(sp);
    const uint64_t cap = (uint64_t)sms_streamed() * kStreamCtasPerSm;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The shard runs as the fused step's launch windows: kernel boundaries
    // keep the SMs at the same place in the rows.
    return for_each_window(g->offset, n, ZERO_FUSED_WINDOW_ELEMS, [&](uint64_t w0, uint64_t w1) {
        StreamArgs s = base;
        s.e0 = w0;
        s.a.g += w0;
        s.a.p_in += w0;
        s.a.m_in += w0;
        s.a.v_in += w0;
        s.a.p_out += w0;
        s.a.m_out += w0;
        s.a.v_out += w0;
        s.a.gath += w0;
        const uint64_t len = w1 - w0;
        const uint64_t head = (8 - ((g->offset + w0) & 7)) & 7;
        s.a.sp.len = len;
        s.a.sp.head = head < len ? head : len;
        s.a.sp.nvec = (len - s.a.sp.head) / 8;
        const uint64_t want = (len / 8 + kStreamThreads - 1) / kStreamThreads;
        const unsigned grid = (unsigned)(want == 0 ? 1 : (want < cap ? want : cap));
#define ZERO_STREAM_LAUNCH(DT, V8)                                                          \
    switch (width) {                                                                        \
    case 16: k_step_streamed<DT, 16, V8><<<grid, kStreamThreads, 0, st>>>(s); break;        \
    case 8: k_step_streamed<DT, 8, V8><<<grid, kStreamThreads, 0, st>>>(s); break;          \
    case 4: k_step_streamed<DT, 4, V8><<<grid, kStreamThreads, 0, st>>>(s); break;          \
    default: k_step_streamed<DT, 2, V8><<<grid, kStreamThreads, 0, st>>>(s); break;         \
    }
        if (g->dtype == ZERO_F16) {
            if (v8) {
                ZERO_STREAM_LAUNCH(ZERO_F16, true)
            } else {
                ZERO_STREAM_LAUNCH(ZERO_F16, false)
            }
        } else {
            if (v8) {
                ZERO_STREAM_LAUNCH(ZERO_BF16, true)
            } else {
                ZERO_STREAM_LAUNCH(ZERO_BF16, false)
            }
        }
#undef ZERO_STREAM_LAUNCH
        return cudaGetLastError() == cudaSuccess ? ZERO_OK : ZERO_ERR_CUDA;
    });
}

extern "C" zero_status_t zero_feed_buckets(const void* host, uint64_t host_row_stride,
                                           const zero_grads_t* g, uint64_t n,
                                           uint64_t bucket_elems, uint32_t* d_ready,
                                           const uint32_t* h_epoch, void* copy_stream)
{
    if (!host || !g || !g->base || g->nd == 0 || !d_ready || !h_epoch || bucket_elems == 0)
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
    const uint64_t nb = (n + bucket_elems - 1) / bucket_elems;
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
