// Device-side building blocks of the ZeRO shard-step kernels (internal).
//
// Included by every CUDA translation unit of the library; everything here is
// __device__ __forceinline__ (or a POD struct) in an anonymous namespace, so
// each translation unit gets its own inlined copy.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "zero.h"
#include "zero_internal.h"

namespace zero {
namespace {

#ifndef ZERO_RANK_UNROLL
#define ZERO_RANK_UNROLL 8
#endif
// L2 prefetch size hint of the ring's cp.async copies (256, 128 or 0 = none).
#ifndef ZERO_CP_ASYNC_L2_HINT
#define ZERO_CP_ASYNC_L2_HINT 256
#endif
constexpr int kRankUnroll = ZERO_RANK_UNROLL;   // rank rows loaded back to back per thread

// ---------------------------------------------------------------------------
// Memory access helpers
// ---------------------------------------------------------------------------

// 16-byte read of gradient data that is used once: bypass L1, hint the L2
// to fetch the whole 256-byte sector group.
__device__ __forceinline__ uint4 ld_grad16(const uint16_t* p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint16_t ld_grad2(const uint16_t* p)
{
    uint16_t r;
    asm("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// 16-byte asynchronous copy global -> shared (L1 bypassed), and its group
// commit / wait.  wait_group is a hardware wait on this thread's own copies.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
#if ZERO_CP_ASYNC_L2_HINT == 256
    asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(sa), "l"(gmem)
                 : "memory");
#elif ZERO_CP_ASYNC_L2_HINT == 128
    asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16;" ::"r"(sa), "l"(gmem)
                 : "memory");
#else
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
#endif
}

__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------------------
// Bulk (TMA) copies and mbarriers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase of parity `parity` of barrier `bar` to complete, for at
// most limit_ns of %globaltimer time (and an iteration cap).  False on expiry.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < (1u << 30); ++i) {
        if (mbar_try_wait(bar, parity))
            return true;
        if ((i & 255) == 255 && global_ns() - t0 > limit_ns)
            return false;
    }
    return false;
}

// Orders this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (bulk copy) accesses to the same memory: a consumer runs it
// after reading a stage and before releasing the stage to be refilled.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// L2 policy for data read exactly once.
__device__ __forceinline__ uint64_t l2_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned)
// global -> this CTA's shared memory; completion is counted as transaction
// bytes on barrier `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Two 16-bit elements packed in a word (element 0 in the low half) to fp32;
// both conversions are exact.
template <int DT>
__device__ __forceinline__ float2 widen2(uint32_t w)
{
    if (DT == ZERO_F16) {
        __half2 h;
        static_assert(sizeof(h) == sizeof(w), "half2 is one word");
        memcpy(&h, &w, sizeof(w));
        return __half22float2(h);
    } else {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    }
}

template <int DT>
__device__ __forceinline__ float widen1(uint16_t b)
{
    if (DT == ZERO_F16)
        return __half2float(__ushort_as_half(b));
    return __uint_as_float((uint32_t)b << 16);
}

// Round-to-nearest-even fp32 -> fp16/bf16 bits.
template <int DT>
__device__ __forceinline__ uint16_t narrow1(float x)
{
    if (DT == ZERO_F16)
        return __half_as_ushort(__float2half_rn(x));
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ bool nonfinite(float x)
{
    return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;   // exponent all ones
}

template <int DT>
__device__ __forceinline__ void set8(float (&a)[8], uint4 w)
{
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = widen2<DT>(ws[i]);
        a[2 * i] = f.x;
        a[2 * i + 1] = f.y;
    }
}

template <int DT>
__device__ __forceinline__ void add8(float (&a)[8], uint4 w)
{
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = widen2<DT>(ws[i]);
        a[2 * i] = __fadd_rn(a[2 * i], f.x);
        a[2 * i + 1] = __fadd_rn(a[2 * i + 1], f.y);
    }
}

// Rank-ordered fold of 8 consecutive elements: acc = ((c_0 + c_1) + ...) +
// c_{nd-1}.  Rows are loaded kRankUnroll at a time so that many 16-byte
// reads are in flight per thread; the adds still run in rank order.
template <int DT>
__device__ __forceinline__ void fold8(const uint16_t* gp, uint64_t row_stride, uint32_t nd,
                                      float (&acc)[8])
{
    set8<DT>(acc, ld_grad16(gp));
    for (uint32_t j0 = 1; j0 < nd; j0 += kRankUnroll) {
        uint4 w[kRankUnroll];
#pragma unroll
        for (int u = 0; u < kRankUnroll; ++u)
            if (j0 + u < nd)
                w[u] = ld_grad16(gp + (uint64_t)(j0 + u) * row_stride);
#pragma unroll
        for (int u = 0; u < kRankUnroll; ++u)
            if (j0 + u < nd)
                add8<DT>(acc, w[u]);
    }
}

template <int DT>
__device__ __forceinline__ float fold1(const uint16_t* gp, uint64_t row_stride, uint32_t nd)
{
    float s = widen1<DT>(ld_grad2(gp));
    for (uint32_t j = 1; j < nd; ++j)
        s = __fadd_rn(s, widen1<DT>(ld_grad2(gp + (uint64_t)j * row_stride)));
    return s;
}

// AdamW on one element (decoupled weight decay, bias correction, eps outside
// the square root), every operation correctly rounded.
__device__ __forceinline__ void adamw1(const StepScalars& k, float g, float& p, float& m,
                                       float& v)
{
    const float m1 = __fadd_rn(__fmul_rn(k.b1, m), __fmul_rn(k.c1, g));
    const float v1 = __fadd_rn(__fmul_rn(k.b2, v), __fmul_rn(k.c2, __fmul_rn(g, g)));
    const float m_hat = __fdiv_rn(m1, k.bc1);
    const float v_hat = __fdiv_rn(v1, k.bc2);
    const float u = __fdiv_rn(m_hat, __fadd_rn(__fsqrt_rn(v_hat), k.eps));
    p = __fsub_rn(__fmul_rn(p, k.wdf), __fmul_rn(k.lr, u));
    m = m1;
    v = v1;
}

// Store 8 consecutive 16-bit values (packed in 4 words) at q, using the
// widest stores the address phase allows (W = 16, 8, 4 or 2 bytes).
template <int W>
__device__ __forceinline__ void store8(uint16_t* q, const uint32_t (&w)[4])
{
    if (W == 16) {
        __stcs(reinterpret_cast<uint4*>(q), make_uint4(w[0], w[1], w[2], w[3]));
    } else if (W == 8) {
        __stcs(reinterpret_cast<uint2*>(q), make_uint2(w[0], w[1]));
        __stcs(reinterpret_cast<uint2*>(q + 4), make_uint2(w[2], w[3]));
    } else if (W == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            __stcs(reinterpret_cast<unsigned int*>(q + 2 * i), w[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __stcs(reinterpret_cast<unsigned short*>(q + 2 * i), (unsigned short)(w[i] & 0xFFFF));
            __stcs(reinterpret_cast<unsigned short*>(q + 2 * i + 1), (unsigned short)(w[i] >> 16));
        }
    }
}

__device__ __forceinline__ void flag_if_any(bool bad, uint32_t* flag)
{
    if (__any_sync(0xFFFFFFFFu, bad) && (threadIdx.x & 31) == 0)
        atomicOr(flag, 1u);
}

// Element split of a window [0, len): `head` scalar elements up to the first
// 16-byte aligned gradient element, `nvec` 8-element vectors, then a scalar
// tail.  Scalar elements are handled by the first threads of the grid.
struct Split {
    uint64_t len;
    uint64_t head;
    uint64_t nvec;
    __host__ __device__ __forceinline__ uint64_t nscalar() const { return len - 8 * nvec; }
    __host__ __device__ __forceinline__ uint64_t scalar_elem(uint64_t t) const
    {
        return t < head ? t : head + 8 * nvec + (t - head);
    }
};

struct FusedArgs {
    const uint16_t* g;     // element 0 of the window in row 0
    uint64_t row_stride;   // elements
    uint32_t nd;
    Split sp;
    const float* p_in;
    const float* m_in;
    const float* v_in;
    float* p_out;
    float* m_out;
    float* v_out;
    uint16_t* gath;        // gathered element of window element 0
    StepScalars k;
    uint32_t* flag;
    const uint32_t* gate;  // if non-null and nonzero at launch, the launch does nothing
    float* cb;             // reduction-only launches: cb[e] = sum * k.inv (null: check only)
    uint32_t early;        // 1: start at once, wait for the predecessor only at the end
};

// First instructions of every step kernel: under a programmatic dependent
// launch, wait until the previous grid in the stream has completed and its
// writes are visible, then let the next grid be scheduled.  No-ops on a
// plain launch.
__device__ __forceinline__ void pdl_entry()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The same for a launch window after the first of one call: its elements are
// disjoint from its predecessor's, so it starts work at once and waits for
// the predecessor only before it ends (pdl_end).  It therefore never
// completes before its predecessor, and a kernel that waits for it also
// waits for every earlier window.
__device__ __forceinline__ void pdl_begin(uint32_t early)
{
    if (!early)
        asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_end(uint32_t early)
{
    if (early)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

// True if the launch is gated off (a bucket wait before it ran out).
__device__ __forceinline__ bool gated(const FusedArgs& a)
{
    return a.gate && *static_cast<const volatile uint32_t*>(a.gate) != 0;
}

// Scalar element e of the window (head or tail): fold, AdamW, cast.
template <int DT>
__device__ __forceinline__ bool fused_scalar(const FusedArgs& a, uint64_t e)
{
    const float s = fold1<DT>(a.g + e, a.row_stride, a.nd);
    float p = a.p_in[e], m = a.m_in[e], v = a.v_in[e];
    adamw1(a.k, __fmul_rn(s, a.k.inv), p, m, v);
    a.p_out[e] = p;
    a.m_out[e] = m;
    a.v_out[e] = v;
    a.gath[e] = narrow1<DT>(p);
    return nonfinite(s);
}

// 32-byte (256-bit) streaming load / store of 8 floats at a 32-byte aligned
// address: one instruction covers a whole L2 sector, so no sector is ever
// left half written.
// 1: the state loads also ask L2 for whole 256-byte blocks (measured +0.5% on
// the 8-row workload, level on the 64-row ones).
#ifndef ZERO_STATE_L2_HINT
#define ZERO_STATE_L2_HINT 1
#endif
__device__ __forceinline__ void ld8_cs(const float* p, float (&x)[8])
{
#if ZERO_STATE_L2_HINT
    asm volatile("ld.global.cs.L2::256B.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]), "=f"(x[4]), "=f"(x[5]),
                   "=f"(x[6]), "=f"(x[7])
                 : "l"(p));
#else
    asm volatile("ld.global.cs.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3]), "=f"(x[4]), "=f"(x[5]),
                   "=f"(x[6]), "=f"(x[7])
                 : "l"(p));
#endif
}

__device__ __forceinline__ void st8_cs(float* p, const float (&x)[8])
{
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
                 "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]), "f"(x[6]),
                 "f"(x[7])
                 : "memory");
}

// Epilogue of 8 reduced sums at window element e: scale, AdamW, streaming
// state stores, cast into the gathered slot.  V8 (state pointers 32-byte
// aligned at e): p, m, v move as one 32-byte access each per thread, which
// writes whole sectors.  Otherwise the state moves as two halves of 4
// elements (16-byte accesses), which also bounds live registers.  Returns
// "any sum nonfinite".
template <int DT, int W, bool V8>
__device__ __forceinline__ bool fused_epilogue(const FusedArgs& a, uint64_t e, const float (&s)[8])
{
    bool bad = false;
    uint32_t out16[4];
    if (V8) {
        float p[8], m[8], v[8];
        ld8_cs(a.p_in + e, p);
        ld8_cs(a.m_in + e, m);
        ld8_cs(a.v_in + e, v);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            bad |= nonfinite(s[i]);
            adamw1(a.k, __fmul_rn(s[i], a.k.inv), p[i], m[i], v[i]);
        }
        st8_cs(a.p_out + e, p);
        st8_cs(a.m_out + e, m);
        st8_cs(a.v_out + e, v);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            out16[i] = (uint32_t)narrow1<DT>(p[2 * i]) | ((uint32_t)narrow1<DT>(p[2 * i + 1]) << 16);
    } else {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float4 pp = __ldcs(reinterpret_cast<const float4*>(a.p_in + e) + h);
            const float4 mm = __ldcs(reinterpret_cast<const float4*>(a.m_in + e) + h);
            const float4 vv = __ldcs(reinterpret_cast<const float4*>(a.v_in + e) + h);
            float p[4] = {pp.x, pp.y, pp.z, pp.w};
            float m[4] = {mm.x, mm.y, mm.z, mm.w};
            float v[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                bad |= nonfinite(s[4 * h + i]);
                adamw1(a.k, __fmul_rn(s[4 * h + i], a.k.inv), p[i], m[i], v[i]);
            }
            __stcs(reinterpret_cast<float4*>(a.p_out + e) + h, make_float4(p[0], p[1], p[2], p[3]));
            __stcs(reinterpret_cast<float4*>(a.m_out + e) + h, make_float4(m[0], m[1], m[2], m[3]));
            __stcs(reinterpret_cast<float4*>(a.v_out + e) + h, make_float4(v[0], v[1], v[2], v[3]));
            out16[2 * h] = (uint32_t)narrow1<DT>(p[0]) | ((uint32_t)narrow1<DT>(p[1]) << 16);
            out16[2 * h + 1] = (uint32_t)narrow1<DT>(p[2]) | ((uint32_t)narrow1<DT>(p[3]) << 16);
        }
    }
    store8<W>(a.gath + e, out16);
    return bad;
}

// Epilogue with the state already loaded (p, m, v of the 8 elements at e,
// read with ld8_cs before the fold): scale, AdamW, 256-bit streaming stores,
// cast into the gathered slot.  Returns "any sum nonfinite".
template <int DT, int W>
__device__ __forceinline__ bool fused_epilogue_loaded(const FusedArgs& a, uint64_t e,
                                                      const float (&s)[8], float (&p)[8],
                                                      float (&m)[8], float (&v)[8])
{
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        bad |= nonfinite(s[i]);
        adamw1(a.k, __fmul_rn(s[i], a.k.inv), p[i], m[i], v[i]);
    }
    st8_cs(a.p_out + e, p);
    st8_cs(a.m_out + e, m);
    st8_cs(a.v_out + e, v);
    uint32_t out16[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        out16[i] = (uint32_t)narrow1<DT>(p[2 * i]) | ((uint32_t)narrow1<DT>(p[2 * i + 1]) << 16);
    store8<W>(a.gath + e, out16);
    return bad;
}

// Calls fn(w0, w1) for ceil(len / max_window) launch windows of about equal
// length (max_window a multiple of 16) covering [0, len) of a range whose
// rows' element 0 has phase `phase` (elements past a 32-byte boundary): every
// cut falls on a 16-element (32-byte, one L2 sector) boundary of the rows, and
// a remainder of under 64 elements joins the last window.  Moving the cuts
// back to those boundaries shortens the first window by the phase and can
// lengthen the last to max_window + 15 elements.  Stops at the
// first status other than ZERO_OK.
template <typename F>
zero_status_t for_each_window(uint64_t phase, uint64_t len, uint64_t max_window, F&& fn)
{
    const uint64_t nwin = (len + max_window - 1) / max_window;
    const uint64_t target = ((len + nwin - 1) / nwin + 15) / 16 * 16;
    uint64_t cut = target - (phase & 15);
    for (uint64_t w0 = 0; w0 < len; cut += target) {
        uint64_t w1 = cut < len ? cut : len;
        if (len - w1 < 64)
            w1 = len;
        const zero_status_t st = fn(w0, w1);
        if (st != ZERO_OK)
            return st;
        w0 = w1;
    }
    return ZERO_OK;
}

// True if every state pointer of the fused step is 32-byte aligned (the
// vectors of every window then are too: they start at multiples of 8
// elements).
inline bool state_v8_ok(const float* const (&p)[6])
{
    for (const float* x : p)
        if (((uintptr_t)x & 31) != 0)
            return false;
    return true;
}

}  // namespace
}  // namespace zero
