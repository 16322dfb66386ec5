// The default fused-step kernel, k_step_fused_ring, with its shape constants
// and reduction-only modes (internal; included by zero_kernels.cu).
//
// The kernel is a persistent grid of one 512-thread CTA per SM that stages
// the Nd contribution rows through a per-thread cp.async ring in shared
// memory and moves the fp32 state with 256-bit streaming accesses.  The same
// loop, with a different epilogue, is the reduction of the unfused path (K1:
// scaled sums into the fusion buffer) and the nonfinite pre-check (K5).
#pragma once

#include "zero_device.cuh"

namespace zero {
namespace {

#ifndef ZERO_RING_ROWS
#define ZERO_RING_ROWS 8
#endif
#ifndef ZERO_RING_DEPTH
#define ZERO_RING_DEPTH 2
#endif
#ifndef ZERO_RING_THREADS
#define ZERO_RING_THREADS 512
#endif
// 1: with 32-byte aligned state, the ring kernel loads a vector's p, m, v when
// it starts folding the vector, so their latency hides behind the fold.  Off
// by default: measured about 1% slower on every workload (the ring already
// keeps the next vector's rows in flight during the epilogue).
#ifndef ZERO_STATE_PREFETCH
#define ZERO_STATE_PREFETCH 0
#endif
constexpr int kRingRows = ZERO_RING_ROWS;
constexpr int kRingDepth = ZERO_RING_DEPTH;
constexpr int kRingThreads = ZERO_RING_THREADS;
constexpr size_t kRingBytes = (size_t)kRingDepth * kRingRows * kRingThreads * 16;
static_assert(kRingBytes <= 227 * 1024, "ring exceeds shared memory");

// Epilogue modes of the ring kernel: the whole step, or the reduction alone
// (K1: scaled sums into the fusion buffer; K5: the nonfinite check).
constexpr int kModeStep = 0;
constexpr int kModeReduce = 1;
constexpr int kModeCheck = 2;

// Reduction-only epilogue of 8 sums at window element e: the nonfinite test,
// and for K1 the scaled sums into cb (VEC: cb + e is 16-byte aligned).
template <int MODE, bool VEC>
__device__ __forceinline__ bool reduce_epilogue(const FusedArgs& a, uint64_t e,
                                                const float (&s)[8])
{
    bool bad = false;
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        bad |= nonfinite(s[i]);
        x[i] = __fmul_rn(s[i], a.k.inv);
    }
    if (MODE == kModeReduce) {
        if (VEC) {
            __stcg(reinterpret_cast<float4*>(a.cb + e), make_float4(x[0], x[1], x[2], x[3]));
            __stcg(reinterpret_cast<float4*>(a.cb + e) + 1, make_float4(x[4], x[5], x[6], x[7]));
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                __stcg(a.cb + e + i, x[i]);
        }
    }
    return bad;
}

// Scalar element e of a reduction-only launch.
template <int DT, int MODE>
__device__ __forceinline__ bool reduce_scalar(const FusedArgs& a, uint64_t e)
{
    const float s = fold1<DT>(a.g + e, a.row_stride, a.nd);
    if (MODE == kModeReduce)
        a.cb[e] = __fmul_rn(s, a.k.inv);
    return nonfinite(s);
}

// K4, ring variant.  Each thread walks its vectors (8 elements) as a stream
// of row groups (kRingRows rows of 16 bytes); group copies are issued
// kRingDepth - 1 groups ahead into the thread's private slots of a shared
// ring, so the next vector's rows are already in flight during a vector's
// epilogue.  Slots are laid out [depth][row][thread] so a warp's 16-byte
// reads are contiguous.  Only the issuing thread reads its slots, so
// cp.async.wait_group needs no block barrier.  Rows are still folded in
// rank order.
template <int DT, int W, bool V8, int MODE = kModeStep>
__global__ void __launch_bounds__(kRingThreads, 1) k_step_fused_ring(const FusedArgs a)
{
    extern __shared__ uint4 ring[];
    pdl_begin(a.early);
    // Gated off: a bucket wait of this call ran out.  Only a wait sets the
    // gate, and every window of a group runs after the group's wait, so
    // either all of the group's windows see it set and write nothing, or none
    // does; returning without the end wait of an early window is then safe.
    if (gated(a))
        return;
    bool bad = false;
    const int t = threadIdx.x;
    const uint64_t tid = (uint64_t)blockIdx.x * kRingThreads + t;
    const uint64_t nthr = (uint64_t)gridDim.x * kRingThreads;
    if (tid < a.sp.nscalar()) {
        if (MODE == kModeStep)
            bad |= fused_scalar<DT>(a, a.sp.scalar_elem(tid));
        else
            bad |= reduce_scalar<DT, MODE>(a, a.sp.scalar_elem(tid));
    }

    const uint32_t groups = (a.nd + kRingRows - 1) / kRingRows;   // groups per vector
    const uint16_t* base = a.g + a.sp.head;
    // issue cursor (vector qi, group gi) and consume cursor (qc, gc)
    uint64_t qi = tid;
    uint32_t gi = 0;
    int slot_i = 0;
    auto issue = [&]() {
        if (qi < a.sp.nvec) {
            const uint16_t* gp = base + 8 * qi;
#pragma unroll
            for (int u = 0; u < kRingRows; ++u) {
                const uint32_t j = gi * kRingRows + u;
                if (j < a.nd)
                    cp_async16(&ring[(slot_i * kRingRows + u) * kRingThreads + t],
                               gp + (uint64_t)j * a.row_stride);
            }
        }
        cp_async_commit();
        slot_i = slot_i + 1 == kRingDepth ? 0 : slot_i + 1;
        if (++gi == groups) {
            gi = 0;
            qi += nthr;
        }
    };
#pragma unroll
    for (int d = 0; d < kRingDepth - 1; ++d)
        issue();
    int slot_c = 0;
    uint32_t gc = 0;
    float acc[8];
    float sp[8], sm[8], sv[8];     // the current vector's state (prefetch mode)
    constexpr bool kPrefetch = MODE == kModeStep && V8 && ZERO_STATE_PREFETCH;
    for (uint64_t qc = tid; qc < a.sp.nvec;) {
        issue();
        cp_async_wait<kRingDepth - 1>();     // the oldest group has landed
        if (kPrefetch && gc == 0) {
            const uint64_t e = a.sp.head + 8 * qc;
            ld8_cs(a.p_in + e, sp);
            ld8_cs(a.m_in + e, sm);
            ld8_cs(a.v_in + e, sv);
        }
#pragma unroll
        for (int u = 0; u < kRingRows; ++u) {
            const uint32_t j = gc * kRingRows + u;
            if (j < a.nd) {
                const uint4 w = ring[(slot_c * kRingRows + u) * kRingThreads + t];
                if (j == 0)
                    set8<DT>(acc, w);
                else
                    add8<DT>(acc, w);
            }
        }
        slot_c = slot_c + 1 == kRingDepth ? 0 : slot_c + 1;
        if (++gc == groups) {
            gc = 0;
            if (MODE != kModeStep)
                bad |= reduce_epilogue<MODE, W == 16>(a, a.sp.head + 8 * qc, acc);
            else if (kPrefetch)
                bad |= fused_epilogue_loaded<DT, W>(a, a.sp.head + 8 * qc, acc, sp, sm, sv);
            else
                bad |= fused_epilogue<DT, W, V8>(a, a.sp.head + 8 * qc, acc);
            qc += nthr;
        }
    }
    cp_async_wait<0>();
    flag_if_any(bad, a.flag);
    pdl_end(a.early);
}

}  // namespace
}  // namespace zero
