// The short-window fused-step kernel, k_step_fused_small, with its two
// compiled shapes (internal; included by zero_kernels.cu).
//
// A launch window that one wave of this kernel covers runs here instead of on
// the ring kernel: each thread takes 4 elements (8-byte row reads, 16-byte
// state accesses), so a short window spreads over every SM.
#pragma once

#include "zero_device.cuh"

namespace zero {
namespace {

// 8-byte read of gradient data used once (4 elements of one row).
__device__ __forceinline__ uint2 ld_grad8(const uint16_t* p)
{
    uint2 r;
    asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

template <int DT>
__device__ __forceinline__ void add4(float (&a)[4], uint2 w, bool first)
{
    const float2 lo = widen2<DT>(w.x), hi = widen2<DT>(w.y);
    if (first) {
        a[0] = lo.x;
        a[1] = lo.y;
        a[2] = hi.x;
        a[3] = hi.y;
    } else {
        a[0] = __fadd_rn(a[0], lo.x);
        a[1] = __fadd_rn(a[1], lo.y);
        a[2] = __fadd_rn(a[2], hi.x);
        a[3] = __fadd_rn(a[3], hi.y);
    }
}

// Store 4 consecutive 16-bit values (packed in 2 words) at q with the widest
// stores its address allows (W = 8, 4 or 2 bytes).
template <int W>
__device__ __forceinline__ void store4(uint16_t* q, uint32_t w0, uint32_t w1)
{
    if (W == 8) {
        __stcs(reinterpret_cast<uint2*>(q), make_uint2(w0, w1));
    } else if (W == 4) {
        __stcs(reinterpret_cast<unsigned int*>(q), w0);
        __stcs(reinterpret_cast<unsigned int*>(q + 2), w1);
    } else {
        __stcs(reinterpret_cast<unsigned short*>(q), (unsigned short)(w0 & 0xFFFF));
        __stcs(reinterpret_cast<unsigned short*>(q + 1), (unsigned short)(w0 >> 16));
        __stcs(reinterpret_cast<unsigned short*>(q + 2), (unsigned short)(w1 & 0xFFFF));
        __stcs(reinterpret_cast<unsigned short*>(q + 3), (unsigned short)(w1 >> 16));
    }
}

// Element split of a short window into 4-element groups: `head` scalar
// elements up to the first row element on an 8-byte boundary, `nquad`
// groups, then a scalar tail (at most 3 + 3 scalar elements in all).
struct QuadSplit {
    uint64_t head;
    uint64_t nquad;
};

constexpr int kSmallThreads = 256;

// The two compiled shapes of the short-window kernel.
//  - wide: 8 rank rows loaded back to back, the state loaded after the fold,
//    80 registers, 3 CTAs a SM;
//  - light: 4 rows back to back, the state loaded before the fold (its
//    latency then hides behind the rows'), at most 64 registers, 4 CTAs a SM.
// Measured over 1 to 64 rows of 65,536 to 466,944 elements (graph-timed
// back-to-back steps): light is up to 22% faster on up to 16 rows while the
// window needs at most 2 CTAs a SM (level on 8 rows of 131,072), wide is
// faster on 64 rows (light up to 31% slower) and once the window fills a wave
// of 3 CTAs a SM.
template <bool LIGHT>
struct SmallShape {
    static constexpr int ctas_per_sm = LIGHT ? 4 : 3;
    static constexpr int unroll = LIGHT ? 4 : 8;
};
// The light shape's limits: rows, and windows of at most this many CTAs a SM.
#ifndef ZERO_SMALL_LIGHT_CTAS
#define ZERO_SMALL_LIGHT_CTAS 2
#endif
constexpr uint32_t kSmallLightMaxNd = 16;
constexpr uint64_t kSmallLightCtasPerSm = ZERO_SMALL_LIGHT_CTAS;

// K4, short-window variant.  A window shorter than one pass of the ring
// kernel's grid leaves most of the ring's threads idle and puts the AdamW
// arithmetic (three correctly rounded divisions and a square root an
// element) on a few SMs; this kernel gives each thread 4 elements (8-byte
// row reads, 16-byte state accesses), so the same window spreads over every
// SM with twice to four times the threads.  Within one wave of its grid
// (3 CTAs a SM) it beat the ring on every shard measured, by 10% (4 rows of
// 262,144) to 46% (64 rows of 65,536); past one wave the ring wins.  The
// fold, the op order and the stores' values are those of every other
// variant.
template <int DT, int W, bool LIGHT>
__global__ void __launch_bounds__(kSmallThreads, SmallShape<LIGHT>::ctas_per_sm)
    k_step_fused_small(const FusedArgs a, const QuadSplit qs)
{
    constexpr int kUnroll = SmallShape<LIGHT>::unroll;
    pdl_begin(a.early);
    if (gated(a))   // all of a group's windows see the gate alike (see k_step_fused_ring)
        return;
    bool bad = false;
    const uint64_t tid = (uint64_t)blockIdx.x * kSmallThreads + threadIdx.x;
    const uint64_t nthr = (uint64_t)gridDim.x * kSmallThreads;
    const uint64_t nscalar = a.sp.len - 4 * qs.nquad;
    if (tid < nscalar)
        bad |= fused_scalar<DT>(a, tid < qs.head ? tid : qs.head + 4 * qs.nquad + (tid - qs.head));
    for (uint64_t q = tid; q < qs.nquad; q += nthr) {
        const uint64_t e = qs.head + 4 * q;
        const uint16_t* gp = a.g + e;
        float4 pp, mm, vv;
        if (LIGHT) {
            pp = __ldcs(reinterpret_cast<const float4*>(a.p_in + e));
            mm = __ldcs(reinterpret_cast<const float4*>(a.m_in + e));
            vv = __ldcs(reinterpret_cast<const float4*>(a.v_in + e));
        }
        float s[4];
        add4<DT>(s, ld_grad8(gp), true);
        for (uint32_t j0 = 1; j0 < a.nd; j0 += kUnroll) {
            uint2 w[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (j0 + u < a.nd)
                    w[u] = ld_grad8(gp + (uint64_t)(j0 + u) * a.row_stride);
#pragma unroll
            for (int u = 0; u < kUnroll; ++u)
                if (j0 + u < a.nd)
                    add4<DT>(s, w[u], false);
        }
        if (!LIGHT) {
            pp = __ldcs(reinterpret_cast<const float4*>(a.p_in + e));
            mm = __ldcs(reinterpret_cast<const float4*>(a.m_in + e));
            vv = __ldcs(reinterpret_cast<const float4*>(a.v_in + e));
        }
        float p[4] = {pp.x, pp.y, pp.z, pp.w};
        float m[4] = {mm.x, mm.y, mm.z, mm.w};
        float v[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            bad |= nonfinite(s[i]);
            adamw1(a.k, __fmul_rn(s[i], a.k.inv), p[i], m[i], v[i]);
        }
        __stcs(reinterpret_cast<float4*>(a.p_out + e), make_float4(p[0], p[1], p[2], p[3]));
        __stcs(reinterpret_cast<float4*>(a.m_out + e), make_float4(m[0], m[1], m[2], m[3]));
        __stcs(reinterpret_cast<float4*>(a.v_out + e), make_float4(v[0], v[1], v[2], v[3]));
        store4<W>(a.gath + e, (uint32_t)narrow1<DT>(p[0]) | ((uint32_t)narrow1<DT>(p[1]) << 16),
                  (uint32_t)narrow1<DT>(p[2]) | ((uint32_t)narrow1<DT>(p[3]) << 16));
    }
    flag_if_any(bad, a.flag);
    pdl_end(a.early);
}

}  // namespace
}  // namespace zero
