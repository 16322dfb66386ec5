// Device kernels and launchers of the ZeRO shard-step C ABI (sm_103a).
//
// One data-parallel rank's partitioned optimizer step ("ZeRO: Memory
// Optimizations Toward Training Trillion Parameter Models", section "ZeRO-DP":
// Stage 2 reduce-scatters gradients bucket by bucket, each rank updates only
// its 1/Nd of the fp32 optimizer state, Stage 1 all-gathers the parameters),
// with the Nd ranks' gradients emulated as Nd rows in this GPU's memory.
//
// The step is elementwise and HBM-bound: at Nd = 64 a parameter costs
// 2*Nd + 26 bytes (Nd 2-byte gradient reads, 12 B of fp32 state read, 12 B
// written, 2 B cast out) for ~Nd + 30 flops, so it is not tensor-core work.
// The fused step (k_step_fused_ring) is a persistent grid of one 512-thread
// CTA per SM that stages the Nd contribution rows through a per-thread
// cp.async ring in shared memory (16-byte copies, two row groups deep) and
// moves the fp32 state with 256-bit streaming accesses; a window short enough
// for one wave of k_step_fused_small (4 elements a thread, zero_small.cuh)
// runs there instead.  Two other variants compute the same step bit for bit:
// k_step_fused (rows loaded straight into registers; the kernel for rows read
// in place from host memory) and k_step_fused_tma (a producer warp's
// cp.async.bulk copies of rows and state into mbarrier-tracked shared-memory
// rings).  The unfused primitives are
// 128-bit grid-stride loops sized to the SM count.
//
// Bit-exactness: every fp32 operation is an explicit correctly rounded
// intrinsic (__fadd_rn/__fmul_rn/__fdiv_rn/__fsqrt_rn), so no multiply-add is
// contracted, and the reduction is a per-element sequential fold over ranks
// 0..Nd-1.  Warp votes are used only for the nonfinite flag.
#include <cuda.h>   // CUcontext and CUresult for two driver queries found at run time
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <utility>

#include "zero_device.cuh"
#include "zero_ring.cuh"
#include "zero_small.cuh"

namespace zero {

zero_status_t resolve_ptr(const void* p, void** out, bool* on_host)
{
    *out = const_cast<void*>(p);
    if (on_host)
        *on_host = false;
    cudaPointerAttributes at;
    const cudaError_t e = cudaPointerGetAttributes(&at, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        // a pointer CUDA does not know is the caller's error; no device or
        // driver is the runtime's
        return e == cudaErrorInvalidValue ? ZERO_ERR_INVALID_ARG : ZERO_ERR_CUDA;
    }
    switch (at.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
        return ZERO_OK;
    case cudaMemoryTypeHost:
        // the mapping keeps the address's place within a 16-byte line, so
        // every alignment the caller's pointer was checked for still holds
        if (!at.devicePointer || (((uintptr_t)at.devicePointer ^ (uintptr_t)p) & 15) != 0)
            return ZERO_ERR_INVALID_ARG;
        *out = at.devicePointer;
        if (on_host)
            *on_host = true;
        return ZERO_OK;
    default:
        return ZERO_ERR_INVALID_ARG;
    }
}

zero_status_t resolve_grads(const zero_grads_t* g, zero_grads_t* out, bool* in_host)
{
    *out = *g;
    void* base = nullptr;
    const zero_status_t st = resolve_ptr(g->base, &base, in_host);
    out->base = base;
    return st;
}

zero_status_t require_device(const void* const* ptrs, int count)
{
    for (int i = 0; i < count; ++i) {
        cudaPointerAttributes at;
        const cudaError_t e = cudaPointerGetAttributes(&at, ptrs[i]);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e == cudaErrorInvalidValue ? ZERO_ERR_INVALID_ARG : ZERO_ERR_CUDA;
        }
        if (at.type != cudaMemoryTypeDevice && at.type != cudaMemoryTypeManaged)
            return ZERO_ERR_INVALID_ARG;
    }
    return ZERO_OK;
}

zero_status_t require_device_state(const zero_state_t* in, const zero_state_t* out,
                                   const void* word)
{
    const void* p[7] = {in->master, in->m, in->v, out->master, out->m, out->v, word};
    return require_device(p, word ? 7 : 6);
}

namespace {

constexpr int kThreads = 256;       // threads per CTA
#ifndef ZERO_CTAS_PER_SM
#define ZERO_CTAS_PER_SM 2
#endif
// Reduction kernels: resident CTAs per SM (2 x 256 threads leaves ~114
// registers a thread, enough for 8 rows of 16-byte loads in flight with no
// spills) and rank rows loaded back to back per thread.
constexpr int kCtasPerSm = ZERO_CTAS_PER_SM;
// Elementwise kernels (AdamW from fp32, cast): full occupancy.
constexpr int kCtasPerSmLight = 8;

// Fused step variant: 0 = rows loaded into registers; 1 = rows staged through
// a per-thread cp.async ring in shared memory (kRingDepth groups of
// kRingRows rows of 16 bytes a thread), which keeps more bytes in flight per
// SM than the register file allows; 2 = rows and state staged by bulk
// copies.  The environment variable ZERO_FUSED_VARIANT ("registers", "ring",
// "tma"), read at each call, overrides this default; every variant gives
// bitwise the same results.
#ifndef ZERO_FUSED_IMPL
#define ZERO_FUSED_IMPL 1
#endif
// Longest launch window of the fused step (elements, a multiple of 16; a
// window can exceed it by the rows' phase within a 32-byte sector plus under
// 64 elements when a range's remainder joins it).
#ifndef ZERO_WINDOW_ELEMS
#define ZERO_WINDOW_ELEMS ZERO_FUSED_WINDOW_ELEMS
#endif
constexpr uint64_t kWindow = ZERO_WINDOW_ELEMS;
static_assert(kWindow % 16 == 0 && kWindow >= 64, "window must be a multiple of 16");

// Fused step, bulk-copy variant (ZERO_FUSED_IMPL 2): a producer warp streams
// each tile's fp32 state (master, m, v) into a 2-slot ring and its rank rows
// into a kTmaStages-deep ring of shared-memory stages, with cp.async.bulk
// (completion counted on each slot's mbarrier); kTmaConsumers consumer
// threads fold the rows, one 8-element vector each per tile, and run the
// epilogue from the staged state.
#ifndef ZERO_TMA_CONSUMERS
#define ZERO_TMA_CONSUMERS 512
#endif
#ifndef ZERO_TMA_ROWS
#define ZERO_TMA_ROWS 4
#endif
#ifndef ZERO_TMA_STAGES
#define ZERO_TMA_STAGES 4
#endif
constexpr int kTmaConsumers = ZERO_TMA_CONSUMERS;
constexpr int kTmaThreads = kTmaConsumers + 32;          // + the producer warp
constexpr int kTmaRows = ZERO_TMA_ROWS;                  // rank rows per stage
constexpr int kTmaStages = ZERO_TMA_STAGES;
constexpr int kTmaStateSlots = 2;
constexpr uint32_t kTmaRowBytes = kTmaConsumers * 16;    // one row of one tile
constexpr size_t kTmaStageBytes = (size_t)kTmaRows * kTmaRowBytes;
constexpr uint32_t kTmaStateArrayBytes = kTmaConsumers * 32;   // 8 floats a consumer
constexpr size_t kTmaStateSlotBytes = 3 * (size_t)kTmaStateArrayBytes;
constexpr size_t kTmaBarOffset = kTmaStages * kTmaStageBytes + kTmaStateSlots * kTmaStateSlotBytes;
constexpr size_t kTmaBytes =
    kTmaBarOffset + 2 * (kTmaStages + kTmaStateSlots) * sizeof(uint64_t);
static_assert(kTmaConsumers % 32 == 0 && kTmaStages <= 32, "TMA pipeline shape");
static_assert(kTmaBytes <= 227 * 1024, "TMA rings exceed shared memory");
static_assert(kTmaStageBytes < (1u << 20) && kTmaStateSlotBytes < (1u << 20),
              "a slot exceeds an mbarrier phase");
// Longest wait on a pipeline barrier before the kernel gives up (a healthy
// wait lasts microseconds), and on each in-flight copy after giving up.
constexpr uint64_t kTmaWaitNs = 10ull * 1000 * 1000 * 1000;
constexpr uint64_t kTmaDrainNs = 1000ull * 1000 * 1000;

// K4, register variant: fused reduce + scale + AdamW + cast, one pass over
// the window; each thread loads kRankUnroll rows of 16 bytes back to back.
template <int DT, int W, bool V8>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) k_step_fused(const FusedArgs a)
{
    pdl_begin(a.early);
    if (gated(a))   // all of a group's windows see the gate alike (see k_step_fused_ring)
        return;
    bool bad = false;
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint64_t nthr = (uint64_t)gridDim.x * kThreads;
    if (tid < a.sp.nscalar())
        bad |= fused_scalar<DT>(a, a.sp.scalar_elem(tid));
    for (uint64_t q = tid; q < a.sp.nvec; q += nthr) {
        const uint64_t e = a.sp.head + 8 * q;
        float s[8];
        fold8<DT>(a.g + e, a.row_stride, a.nd, s);
        bad |= fused_epilogue<DT, W, V8>(a, e, s);
    }
    flag_if_any(bad, a.flag);
    pdl_end(a.early);
}

// Epilogue of the bulk-copy variant: the state of the 8 elements at e was
// staged in shared memory; the new state leaves with streaming stores
// (32-byte when V8, else two 16-byte halves).  Returns "any sum nonfinite".
template <int DT, int W, bool V8>
__device__ __forceinline__ bool tma_epilogue(const FusedArgs& a, uint64_t e, const float (&s)[8],
                                             float (&p)[8], float (&m)[8], float (&v)[8])
{
    bool bad = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        bad |= nonfinite(s[i]);
        adamw1(a.k, __fmul_rn(s[i], a.k.inv), p[i], m[i], v[i]);
    }
    if (V8) {
        st8_cs(a.p_out + e, p);
        st8_cs(a.m_out + e, m);
        st8_cs(a.v_out + e, v);
    } else {
        float* outs[3] = {a.p_out + e, a.m_out + e, a.v_out + e};
        const float* vals[3] = {p, m, v};
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            __stcs(reinterpret_cast<float4*>(outs[k]),
                   make_float4(vals[k][0], vals[k][1], vals[k][2], vals[k][3]));
            __stcs(reinterpret_cast<float4*>(outs[k]) + 1,
                   make_float4(vals[k][4], vals[k][5], vals[k][6], vals[k][7]));
        }
    }
    uint32_t out16[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        out16[i] = (uint32_t)narrow1<DT>(p[2 * i]) | ((uint32_t)narrow1<DT>(p[2 * i + 1]) << 16);
    store8<W>(a.gath + e, out16);
    return bad;
}

// K4, bulk-copy variant.  Tiles of kTmaConsumers vectors are dealt to the
// CTAs round robin, so the grid moves through the rows together.  For each
// tile the producer thread first copies the tile's master, m and v into a
// state slot, then its rank rows, kTmaRows at a time, into the stage ring.  A
// slot or stage is refilled once all consumers arrived on its "empty"
// barrier; its "full" barrier completes when the copies' bytes have landed.
// Consumers fold the rows in rank order and release each stage, then take
// their vector's state from the slot, release it, and store the new state
// (256-bit streaming stores when 32-byte aligned) and the cast parameters.
// Every barrier wait is bounded: on expiry ZERO_STEP_FLAG_WAIT_TIMEOUT is set
// in the flag word, the producer waits (bounded) for the copies it issued,
// and the CTA ends.
template <int DT, int W, bool V8>
__global__ void __launch_bounds__(kTmaThreads, 1) k_step_fused_tma(const FusedArgs a)
{
    extern __shared__ __align__(128) unsigned char tma_smem[];
    const uint4* stages = reinterpret_cast<const uint4*>(tma_smem);   // [stage][row][consumer]
    const float* slots =                                              // [slot][array][consumer][8]
        reinterpret_cast<const float*>(tma_smem + kTmaStages * kTmaStageBytes);
    uint64_t* bars = reinterpret_cast<uint64_t*>(tma_smem + kTmaBarOffset);
    pdl_begin(a.early);
    // uniform: every thread returns before any barrier; all of a group's
    // windows see the gate alike (see k_step_fused_ring)
    if (gated(a))
        return;
    const uint32_t full0 = smem_u32(bars);                                    // + 8 s
    const uint32_t empty0 = smem_u32(bars + kTmaStages);                      // + 8 s
    const uint32_t sfull0 = smem_u32(bars + 2 * kTmaStages);                  // + 8 slot
    const uint32_t sempty0 = smem_u32(bars + 2 * kTmaStages + kTmaStateSlots);
    const int t = threadIdx.x;
    if (t == 0) {
        for (int s = 0; s < kTmaStages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kTmaConsumers);
        }
        for (int s = 0; s < kTmaStateSlots; ++s) {
            mbar_init(sfull0 + 8 * s, 1);
            mbar_init(sempty0 + 8 * s, kTmaConsumers);
        }
        mbar_fence_init();
    }
    __syncthreads();
    const uint32_t groups = (a.nd + kTmaRows - 1) / kTmaRows;
    const uint64_t ntiles = (a.sp.nvec + kTmaConsumers - 1) / kTmaConsumers;

    if (t >= kTmaConsumers) {                             // producer warp: one thread issues
        if (t != kTmaConsumers)
            return;
        const uint64_t pol = l2_evict_first();
        const uint16_t* base = a.g + a.sp.head;
        const float* state_in[3] = {a.p_in + a.sp.head, a.m_in + a.sp.head, a.v_in + a.sp.head};
        int stage = 0, slot = 0;
        uint32_t phase = 0, sphase = 0;
        uint32_t armed = 0, armed_parity = 0, sarmed = 0, sarmed_parity = 0;
        bool ok = true;
        for (uint64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
            const uint64_t q0 = tile * kTmaConsumers;
            const uint64_t left = a.sp.nvec - q0;
            const uint32_t nv = (uint32_t)(left < (uint64_t)kTmaConsumers ? left : kTmaConsumers);
            // the tile's state
            if (!mbar_wait(sempty0 + 8 * slot, sphase ^ 1, kTmaWaitNs)) {
                ok = false;
                break;
            }
            const uint32_t sfull = sfull0 + 8 * slot;
            mbar_arrive_expect_tx(sfull, 3 * nv * 32);
            const uint32_t sdst = smem_u32(slots + (size_t)slot * 3 * kTmaConsumers * 8);
            for (int k = 0; k < 3; ++k)
                bulk_g2s(sdst + k * kTmaStateArrayBytes, state_in[k] + 8 * q0, nv * 32, sfull,
                         pol);
            sarmed |= 1u << slot;
            sarmed_parity = (sarmed_parity & ~(1u << slot)) | (sphase << slot);
            if (++slot == kTmaStateSlots) {
                slot = 0;
                sphase ^= 1;
            }
            // its rank rows
            const uint32_t bytes = nv * 16;
            const uint16_t* src = base + 8 * q0;
            for (uint32_t gi = 0; gi < groups; ++gi) {
                if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, kTmaWaitNs)) {
                    ok = false;
                    break;
                }
                const uint32_t j0 = gi * kTmaRows;
                const uint32_t rows = a.nd - j0 < (uint32_t)kTmaRows ? a.nd - j0 : kTmaRows;
                const uint32_t full = full0 + 8 * stage;
                mbar_arrive_expect_tx(full, rows * bytes);
                const uint32_t dst = smem_u32(stages + (size_t)stage * kTmaRows * kTmaConsumers);
                for (uint32_t r = 0; r < rows; ++r)
                    bulk_g2s(dst + r * kTmaRowBytes, src + (uint64_t)(j0 + r) * a.row_stride,
                             bytes, full, pol);
                armed |= 1u << stage;
                armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == kTmaStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if (!ok) {
            atomicOr(a.flag, ZERO_STEP_FLAG_WAIT_TIMEOUT);
            for (int s = 0; s < kTmaStages; ++s)      // copies still in flight land first
                if ((armed >> s) & 1)
                    (void)mbar_wait(full0 + 8 * s, (armed_parity >> s) & 1, kTmaDrainNs);
            for (int s = 0; s < kTmaStateSlots; ++s)
                if ((sarmed >> s) & 1)
                    (void)mbar_wait(sfull0 + 8 * s, (sarmed_parity >> s) & 1, kTmaDrainNs);
        }
        pdl_end(a.early);
        return;
    }

    // consumers
    bool bad = false;
    const uint64_t gid = (uint64_t)blockIdx.x * kTmaConsumers + t;
    if (gid < a.sp.nscalar())
        bad |= fused_scalar<DT>(a, a.sp.scalar_elem(gid));
    int stage = 0, slot = 0;
    uint32_t phase = 0, sphase = 0;
    bool ok = true;
    for (uint64_t tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const uint64_t q = tile * kTmaConsumers + t;
        const bool mine = q < a.sp.nvec;
        float acc[8];
        for (uint32_t gi = 0; gi < groups; ++gi) {
            if (!mbar_wait(full0 + 8 * stage, phase, kTmaWaitNs)) {
                ok = false;
                break;
            }
            if (mine) {
                const uint4* row = stages + (size_t)stage * kTmaRows * kTmaConsumers + t;
#pragma unroll
                for (int r = 0; r < kTmaRows; ++r) {
                    const uint32_t j = gi * kTmaRows + r;
                    if (j < a.nd) {
                        const uint4 w = row[r * kTmaConsumers];
                        if (j == 0)
                            set8<DT>(acc, w);
                        else
                            add8<DT>(acc, w);
                    }
                }
            }
            fence_proxy_async_smem();       // reads done before the stage is refilled
            mbar_arrive(empty0 + 8 * stage);
            if (++stage == kTmaStages) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (!ok || !mbar_wait(sfull0 + 8 * slot, sphase, kTmaWaitNs)) {
            ok = false;
            break;
        }
        float st[3][8];
        if (mine) {
            const float* sl = slots + (size_t)slot * 3 * kTmaConsumers * 8 + 8 * t;
#pragma unroll
            for (int k = 0; k < 3; ++k) {
                const float4 lo = *reinterpret_cast<const float4*>(sl + k * kTmaConsumers * 8);
                const float4 hi = *reinterpret_cast<const float4*>(sl + k * kTmaConsumers * 8 + 4);
                st[k][0] = lo.x, st[k][1] = lo.y, st[k][2] = lo.z, st[k][3] = lo.w;
                st[k][4] = hi.x, st[k][5] = hi.y, st[k][6] = hi.z, st[k][7] = hi.w;
            }
        }
        fence_proxy_async_smem();
        mbar_arrive(sempty0 + 8 * slot);
        if (++slot == kTmaStateSlots) {
            slot = 0;
            sphase ^= 1;
        }
        if (mine)
            bad |= tma_epilogue<DT, W, V8>(a, a.sp.head + 8 * q, acc, st[0], st[1], st[2]);
    }
    if (!ok)
        atomicOr(a.flag, ZERO_STEP_FLAG_WAIT_TIMEOUT);
    flag_if_any(bad, a.flag);
    pdl_end(a.early);   // the producer and the consumers wait; the CTA outlives neither
}

struct ReduceArgs {
    const uint16_t* g;
    uint64_t row_stride;
    uint32_t nd;
    Split sp;
    float inv;
    float* cb;             // cb[i] for window element i (nullptr: check only)
    uint32_t* flag;
    uint32_t early;        // as FusedArgs::early
};

// K1 (cb != nullptr): reduce-scatter of one bucket into the fusion buffer.
// K5 (cb == nullptr): the nonfinite pre-check, gradients read only.
// VEC: cb + head is 16-byte aligned, so the body stores float4s.
template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) k_reduce(const ReduceArgs a)
{
    pdl_begin(a.early);
    bool bad = false;
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint64_t nthr = (uint64_t)gridDim.x * kThreads;
    if (tid < a.sp.nscalar()) {
        const uint64_t e = a.sp.scalar_elem(tid);
        const float s = fold1<DT>(a.g + e, a.row_stride, a.nd);
        bad |= nonfinite(s);
        if (a.cb)
            a.cb[e] = __fmul_rn(s, a.inv);
    }
    for (uint64_t q = tid; q < a.sp.nvec; q += nthr) {
        const uint64_t e = a.sp.head + 8 * q;
        float s[8];
        fold8<DT>(a.g + e, a.row_stride, a.nd, s);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            bad |= nonfinite(s[i]);
            s[i] = __fmul_rn(s[i], a.inv);
        }
        if (a.cb) {
            if (VEC) {
                __stcg(reinterpret_cast<float4*>(a.cb + e), make_float4(s[0], s[1], s[2], s[3]));
                __stcg(reinterpret_cast<float4*>(a.cb + e) + 1, make_float4(s[4], s[5], s[6], s[7]));
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    __stcg(a.cb + e + i, s[i]);
            }
        }
    }
    flag_if_any(bad, a.flag);
    pdl_end(a.early);
}

struct AdamArgs {
    const float* g;
    const float* p_in;
    const float* m_in;
    const float* v_in;
    float* p_out;
    float* m_out;
    float* v_out;
    uint64_t n;
    uint64_t head;         // scalar elements before the common 16-byte phase (VEC)
    uint64_t nvec;         // 4-element vectors (VEC)
    StepScalars k;
};

// K2: AdamW from an fp32 reduced gradient.  VEC: every pointer shares one
// 16-byte phase, so the body runs on float4s; otherwise all elements scalar.
template <bool VEC>
__global__ void __launch_bounds__(kThreads, kCtasPerSmLight) k_adam(const AdamArgs a)
{
    pdl_entry();
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint64_t nthr = (uint64_t)gridDim.x * kThreads;
    if (!VEC) {
        for (uint64_t e = tid; e < a.n; e += nthr) {
            float p = a.p_in[e], m = a.m_in[e], v = a.v_in[e];
            adamw1(a.k, a.g[e], p, m, v);
            a.p_out[e] = p;
            a.m_out[e] = m;
            a.v_out[e] = v;
        }
        return;
    }
    const uint64_t nscalar = a.n - 4 * a.nvec;
    if (tid < nscalar) {
        const uint64_t e = tid < a.head ? tid : a.head + 4 * a.nvec + (tid - a.head);
        float p = a.p_in[e], m = a.m_in[e], v = a.v_in[e];
        adamw1(a.k, a.g[e], p, m, v);
        a.p_out[e] = p;
        a.m_out[e] = m;
        a.v_out[e] = v;
    }
    for (uint64_t q = tid; q < a.nvec; q += nthr) {
        const uint64_t e = a.head + 4 * q;
        const float4 gg = __ldcs(reinterpret_cast<const float4*>(a.g + e));
        float4 pp = __ldcs(reinterpret_cast<const float4*>(a.p_in + e));
        float4 mm = __ldcs(reinterpret_cast<const float4*>(a.m_in + e));
        float4 vv = __ldcs(reinterpret_cast<const float4*>(a.v_in + e));
        adamw1(a.k, gg.x, pp.x, mm.x, vv.x);
        adamw1(a.k, gg.y, pp.y, mm.y, vv.y);
        adamw1(a.k, gg.z, pp.z, mm.z, vv.z);
        adamw1(a.k, gg.w, pp.w, mm.w, vv.w);
        __stcs(reinterpret_cast<float4*>(a.p_out + e), pp);
        __stcs(reinterpret_cast<float4*>(a.m_out + e), mm);
        __stcs(reinterpret_cast<float4*>(a.v_out + e), vv);
    }
}

struct CastArgs {
    const float* master;
    uint16_t* gath;        // gathered element of master[0]
    uint64_t n;
    uint64_t head;         // scalar elements until master is 16-byte aligned
    uint64_t nvec;         // 8-element vectors
};

// K3: round-to-nearest-even cast of master weights into the gathered slot.
template <int DT, int W>
__global__ void __launch_bounds__(kThreads, kCtasPerSmLight) k_cast(const CastArgs a)
{
    pdl_entry();
    const uint64_t tid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint64_t nthr = (uint64_t)gridDim.x * kThreads;
    const uint64_t nscalar = a.n - 8 * a.nvec;
    if (tid < nscalar) {
        const uint64_t e = tid < a.head ? tid : a.head + 8 * a.nvec + (tid - a.head);
        a.gath[e] = narrow1<DT>(a.master[e]);
    }
    for (uint64_t q = tid; q < a.nvec; q += nthr) {
        const uint64_t e = a.head + 8 * q;
        const float4 x0 = __ldcs(reinterpret_cast<const float4*>(a.master + e));
        const float4 x1 = __ldcs(reinterpret_cast<const float4*>(a.master + e) + 1);
        const uint32_t w[4] = {
            (uint32_t)narrow1<DT>(x0.x) | ((uint32_t)narrow1<DT>(x0.y) << 16),
            (uint32_t)narrow1<DT>(x0.z) | ((uint32_t)narrow1<DT>(x0.w) << 16),
            (uint32_t)narrow1<DT>(x1.x) | ((uint32_t)narrow1<DT>(x1.y) << 16),
            (uint32_t)narrow1<DT>(x1.z) | ((uint32_t)narrow1<DT>(x1.w) << 16)};
        store8<W>(a.gath + e, w);
    }
}

// ---------------------------------------------------------------------------
// Host-side helpers
// ---------------------------------------------------------------------------

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

// 2-byte elements from the last 32-byte boundary to p: the phase for which
// for_each_window puts every cut on a 32-byte sector boundary of the row.
uint64_t elem_phase(const uint16_t* p) { return ((uintptr_t)p & 31) / 2; }

// Widest store (16/8/4/2 bytes) that a 16-bit element address allows.
int store_width(const void* p)
{
    const uintptr_t x = (uintptr_t)p;
    if ((x & 15) == 0) return 16;
    if ((x & 7) == 0) return 8;
    if ((x & 3) == 0) return 4;
    return 2;
}

int sm_count();

unsigned grid_for(uint64_t work_items, int ctas_per_sm = kCtasPerSm)
{
    const int sms = sm_count();
    const uint64_t want = (work_items + kThreads - 1) / kThreads;
    const uint64_t cap = (uint64_t)sms * ctas_per_sm;
    const uint64_t g = want < cap ? want : cap;
    return (unsigned)(g == 0 ? 1 : g);
}

zero_status_t launch_status()
{
    return cudaGetLastError() == cudaSuccess ? ZERO_OK : ZERO_ERR_CUDA;
}

// Window split for 2-byte gradient rows whose element 0 has phase `phase`
// (elements past a 16-byte boundary).
Split split_window(uint64_t phase, uint64_t len)
{
    Split s;
    s.len = len;
    uint64_t head = (8 - (phase & 7)) & 7;
    s.head = head < len ? head : len;
    s.nvec = (len - s.head) / 8;
    return s;
}

bool mul_overflows(uint64_t a, uint64_t b) { return a != 0 && b > UINT64_MAX / a; }

// Validates a gradient descriptor for elements [begin, begin + n) of the shard.
zero_status_t check_grads(const zero_grads_t* g, uint64_t begin, uint64_t n)
{
    // nd <= ZERO_MAX_ND keeps the kernels' 32-bit row counts (nd + 7,
    // j0 += 8) far from wrapping
    if (!g || !g->base || g->nd == 0 || g->nd > ZERO_MAX_ND ||
        (g->dtype != ZERO_F16 && g->dtype != ZERO_BF16))
        return ZERO_ERR_INVALID_ARG;
    if (!aligned(g->base, 16) || (g->row_stride & 7) != 0 || (g->offset & 7) != 0)
        return ZERO_ERR_ALIGNMENT;
    // the last element read, (nd-1)*row_stride + offset + begin + n, must fit
    if (mul_overflows(g->nd - 1, g->row_stride))
        return ZERO_ERR_INVALID_ARG;
    const uint64_t last_row = (uint64_t)(g->nd - 1) * g->row_stride;
    if (g->offset > UINT64_MAX - last_row || begin > UINT64_MAX - last_row - g->offset ||
        n > UINT64_MAX - last_row - g->offset - begin)
        return ZERO_ERR_INVALID_ARG;
    const uint64_t end = last_row + g->offset + begin + n;
    if (end > (UINT64_MAX >> 1))
        return ZERO_ERR_INVALID_ARG;
    return ZERO_OK;
}

bool ranges_overlap(const void* a, const void* b, uint64_t bytes)
{
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + bytes && y < x + bytes;
}

// in/out state checks: non-null, 16-byte aligned; each output equal to its
// input or disjoint from every input; outputs pairwise disjoint.
zero_status_t check_state(const zero_state_t* in, const zero_state_t* out, uint64_t n,
                          uintptr_t align)
{
    if (!in || !out || !in->master || !in->m || !in->v || !out->master || !out->m || !out->v)
        return ZERO_ERR_INVALID_ARG;
    const float* ins[3] = {in->master, in->m, in->v};
    const float* outs[3] = {out->master, out->m, out->v};
    for (int i = 0; i < 3; ++i)
        if (!aligned(ins[i], align) || !aligned(outs[i], align))
            return ZERO_ERR_ALIGNMENT;
    if (mul_overflows(n, 4))
        return ZERO_ERR_INVALID_ARG;
    const uint64_t bytes = n * 4;
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 3; ++j) {
            if (i == j && outs[i] == ins[j])
                continue;
            if (ranges_overlap(outs[i], ins[j], bytes))
                return ZERO_ERR_INVALID_ARG;
        }
        for (int j = i + 1; j < 3; ++j)
            if (ranges_overlap(outs[i], outs[j], bytes))
                return ZERO_ERR_INVALID_ARG;
    }
    return ZERO_OK;
}

int sm_count()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        sms = 1;
    return sms;
}

// The fused-step variant of a call: ZERO_FUSED_VARIANT if set, else the
// build's default, which with the ring kernel is kVariantAuto: the ring, and
// the short-window kernel for windows that one wave of its grid covers
// (ZERO_SMALL_WINDOWS 0 turns that off).  The ring kernel streams
// HBM-resident rows best.  Rows read in place from host memory always go to
// the register kernel, whose loads keep the host link busier (about 203
// against 183 GB/s on the 7.5B shard's 64 rows).
#ifndef ZERO_SMALL_WINDOWS
#define ZERO_SMALL_WINDOWS 1
#endif
constexpr int kVariantSmall = 3;
constexpr int kVariantAuto = -1;

int fused_variant(bool host_rows)
{
    if (host_rows)
        return 0;
    const char* v = getenv("ZERO_FUSED_VARIANT");
    if (v && strcmp(v, "registers") == 0)
        return 0;
    if (v && strcmp(v, "ring") == 0)
        return 1;
    if (v && strcmp(v, "tma") == 0)
        return 2;
    if (v && strcmp(v, "small") == 0)
        return kVariantSmall;
    return ZERO_FUSED_IMPL == 1 && ZERO_SMALL_WINDOWS ? kVariantAuto : ZERO_FUSED_IMPL;
}

// Elements one wave of the short-window kernel's wide shape covers (3 CTAs a
// SM, 4 elements a thread): a window of at most this many goes to that
// kernel under kVariantAuto.
uint64_t small_window_limit()
{
    return (uint64_t)sm_count() * SmallShape<false>::ctas_per_sm * kSmallThreads * 4;
}

// Opts kernel `fn` in to `bytes` of dynamic shared memory on the current
// device, once per device (a per-device function attribute).  `done` holds a
// bit per device id below 64; higher ids set it on every launch.
template <typename F>
void smem_opt_in(F* fn, size_t bytes, std::atomic<uint64_t>& done)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        dev = 64;
    const uint64_t bit = dev < 64 ? 1ull << dev : 0;
    if (bit && (done.load(std::memory_order_relaxed) & bit))
        return;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
            cudaSuccess && bit)
        done.fetch_or(bit, std::memory_order_relaxed);
}

// Programmatic dependent launch of the ring kernel (on unless ZERO_PDL=0 in
// the environment, read at each call): the next launch in the stream is
// scheduled while this one's last CTAs drain, and waits in the kernel (not
// at the launch) for its predecessor's results.  Consecutive windows and
// steps lose their launch gap: +2% on the 7.5B shard's step.  A window
// after the first of one call works on elements disjoint from its
// predecessor's, so it waits for the predecessor only before it ends
// (pdl_begin / pdl_end with FusedArgs::early): its CTAs start as the
// previous window drains, another +0.7% on that step.  Behind a bucket-ready
// wait this still holds: the first window waits at entry for the wait
// kernel, and a later window is scheduled only after every CTA of the first
// has passed that wait, so the wait has completed (and its status word is
// written) before a later window reads its gate.
bool pdl_enabled()
{
    const char* v = getenv("ZERO_PDL");
    return !(v && v[0] == '0' && v[1] == '\0');
}

// Launches `kern` as a programmatic dependent launch when enabled (every
// step kernel starts with pdl_entry), else as a plain launch.
template <typename... KArgs, typename... Args>
void launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
              Args&&... args)
{
    if (pdl_enabled()) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
    } else {
        kern<<<grid, block, smem, s>>>(std::forward<Args>(args)...);
    }
}

// The shared-memory opt-in of one ring / bulk-copy kernel instance (once
// per device).
template <int DT, int W, bool V8, int MODE>
void ring_opt_in()
{
    static std::atomic<uint64_t> opted{0};
    smem_opt_in(k_step_fused_ring<DT, W, V8, MODE>, kRingBytes, opted);
}

template <int DT, int W, bool V8>
void tma_opt_in()
{
    static std::atomic<uint64_t> opted{0};
    smem_opt_in(k_step_fused_tma<DT, W, V8>, kTmaBytes, opted);
}

template <int DT, int W, bool V8, int MODE>
void launch_ring(unsigned grid, const FusedArgs& a, cudaStream_t s)
{
    ring_opt_in<DT, W, V8, MODE>();
    launch_k(k_step_fused_ring<DT, W, V8, MODE>, dim3(grid), dim3(kRingThreads), kRingBytes, s,
             a);
}

template <int DT, int W, bool V8>
void launch_fused_w(const FusedArgs& a, int variant, cudaStream_t s)
{
    const uint64_t work = a.sp.nvec > a.sp.nscalar() ? a.sp.nvec : a.sp.nscalar();
    if (variant == 2) {
        tma_opt_in<DT, W, V8>();
        const uint64_t tiles = (a.sp.nvec + kTmaConsumers - 1) / kTmaConsumers;
        const uint64_t cap = (uint64_t)sm_count();
        const unsigned grid = (unsigned)(tiles < cap ? (tiles ? tiles : 1) : cap);
        launch_k(k_step_fused_tma<DT, W, V8>, dim3(grid), dim3(kTmaThreads), kTmaBytes, s, a);
    } else if (variant == 1) {
        // one resident CTA per SM; the ring needs the opt-in shared memory size
        const uint64_t want = (work + kRingThreads - 1) / kRingThreads;
        const uint64_t cap = (uint64_t)sm_count();
        const unsigned grid = (unsigned)(want < cap ? (want ? want : 1) : cap);
        launch_ring<DT, W, V8, kModeStep>(grid, a, s);
    } else {
        launch_k(k_step_fused<DT, W, V8>, dim3(grid_for(work)), dim3(kThreads), 0, s, a);
    }
}

template <int DT, bool LIGHT>
void launch_small_shape(const FusedArgs& a, const QuadSplit& qs, uint64_t want, int sms,
                        cudaStream_t s)
{
    const uint64_t cap = (uint64_t)sms * SmallShape<LIGHT>::ctas_per_sm;
    const dim3 grid((unsigned)(want < cap ? (want ? want : 1) : cap));
    const dim3 block(kSmallThreads);
    switch (store_width(a.gath + qs.head)) {
    case 16:
    case 8: launch_k(k_step_fused_small<DT, 8, LIGHT>, grid, block, 0, s, a, qs); break;
    case 4: launch_k(k_step_fused_small<DT, 4, LIGHT>, grid, block, 0, s, a, qs); break;
    default: launch_k(k_step_fused_small<DT, 2, LIGHT>, grid, block, 0, s, a, qs); break;
    }
}

// The short-window kernel over one window: quad split from the rows' phase,
// store width from the gathered slot's (at most 8 bytes), a CTA for every 256
// groups up to one wave (then a grid-stride loop), and the light shape for up
// to 16 rows while the window needs at most 2 CTAs a SM.
template <int DT>
void launch_small(const FusedArgs& a, uint64_t row_phase, cudaStream_t s)
{
    QuadSplit qs;
    const uint64_t head = (4 - (row_phase & 3)) & 3;
    qs.head = head < a.sp.len ? head : a.sp.len;
    qs.nquad = (a.sp.len - qs.head) / 4;
    const uint64_t nscalar = a.sp.len - 4 * qs.nquad;
    const uint64_t work = qs.nquad > nscalar ? qs.nquad : nscalar;
    const uint64_t want = (work + kSmallThreads - 1) / kSmallThreads;
    const int sms = sm_count();
    if (a.nd <= kSmallLightMaxNd && want <= (uint64_t)sms * kSmallLightCtasPerSm)
        launch_small_shape<DT, true>(a, qs, want, sms, s);
    else
        launch_small_shape<DT, false>(a, qs, want, sms, s);
}

template <int DT, bool V8>
void launch_fused_v(const FusedArgs& a, int width, int variant, cudaStream_t s)
{
    switch (width) {
    case 16: launch_fused_w<DT, 16, V8>(a, variant, s); break;
    case 8: launch_fused_w<DT, 8, V8>(a, variant, s); break;
    case 4: launch_fused_w<DT, 4, V8>(a, variant, s); break;
    default: launch_fused_w<DT, 2, V8>(a, variant, s); break;
    }
}

template <int DT>
void launch_fused_dt(const FusedArgs& a, int width, bool v8, int variant, cudaStream_t s)
{
    if (v8)
        launch_fused_v<DT, true>(a, width, variant, s);
    else
        launch_fused_v<DT, false>(a, width, variant, s);
}

template <int DT, bool VEC, int MODE>
void launch_reduce_ring(const FusedArgs& a, cudaStream_t s)
{
    const uint64_t work = a.sp.nvec > a.sp.nscalar() ? a.sp.nvec : a.sp.nscalar();
    const uint64_t want = (work + kRingThreads - 1) / kRingThreads;
    const uint64_t cap = (uint64_t)sm_count();
    const unsigned grid = (unsigned)(want < cap ? (want ? want : 1) : cap);
    launch_ring<DT, VEC ? 16 : 4, false, MODE>(grid, a, s);
}

// K1 (a.cb != nullptr) or K5 over one window: the ring kernel's reduction
// modes, or the register kernel k_reduce for the register variant.
void launch_reduce(const ReduceArgs& r, int dtype, int variant, cudaStream_t s)
{
    const bool vec = r.cb == nullptr || aligned(r.cb + r.sp.head, 16);
    if (variant == 0) {
        const unsigned grid = grid_for(r.sp.nvec > r.sp.nscalar() ? r.sp.nvec : r.sp.nscalar());
        if (dtype == ZERO_F16) {
            if (vec) launch_k(k_reduce<ZERO_F16, true>, dim3(grid), dim3(kThreads), 0, s, r);
            else launch_k(k_reduce<ZERO_F16, false>, dim3(grid), dim3(kThreads), 0, s, r);
        } else {
            if (vec) launch_k(k_reduce<ZERO_BF16, true>, dim3(grid), dim3(kThreads), 0, s, r);
            else launch_k(k_reduce<ZERO_BF16, false>, dim3(grid), dim3(kThreads), 0, s, r);
        }
        return;
    }
    FusedArgs a{};
    a.g = r.g;
    a.row_stride = r.row_stride;
    a.nd = r.nd;
    a.sp = r.sp;
    a.k.inv = r.inv;
    a.flag = r.flag;
    a.cb = r.cb;
    a.early = r.early;
#define ZERO_REDUCE_RING(DT)                                                         \
    if (r.cb && vec) launch_reduce_ring<DT, true, kModeReduce>(a, s);                 \
    else if (r.cb) launch_reduce_ring<DT, false, kModeReduce>(a, s);                  \
    else launch_reduce_ring<DT, true, kModeCheck>(a, s);
    if (dtype == ZERO_F16) {
        ZERO_REDUCE_RING(ZERO_F16)
    } else {
        ZERO_REDUCE_RING(ZERO_BF16)
    }
#undef ZERO_REDUCE_RING
}

void launch_adam(const float* grad, const zero_state_t* in, const zero_state_t* out, uint64_t n,
                 const StepScalars& k, cudaStream_t s)
{
    AdamArgs a{grad, in->master, in->m, in->v, out->master, out->m, out->v, n, 0, 0, k};
    const uintptr_t ph = (uintptr_t)grad & 15;
    const void* ptrs[6] = {in->master, in->m, in->v, out->master, out->m, out->v};
    bool vec = (ph & 3) == 0;
    for (const void* p : ptrs)
        vec = vec && (((uintptr_t)p & 15) == ph);
    if (vec) {
        const uint64_t head = ((16 - ph) & 15) / 4;
        a.head = head < n ? head : n;
        a.nvec = (n - a.head) / 4;
        const uint64_t ns = n - 4 * a.nvec;
        launch_k(k_adam<true>, dim3(grid_for(a.nvec > ns ? a.nvec : ns, kCtasPerSmLight)),
                 dim3(kThreads), 0, s, a);
    } else {
        launch_k(k_adam<false>, dim3(grid_for(n, kCtasPerSmLight)), dim3(kThreads), 0, s, a);
    }
}

void launch_cast(const float* master, uint64_t n, uint16_t* gath, int dtype, cudaStream_t s)
{
    CastArgs a{master, gath, n, 0, 0};
    const uint64_t head = (((16 - ((uintptr_t)master & 15)) & 15) / 4);
    a.head = head < n ? head : n;
    a.nvec = (n - a.head) / 8;
    const uint64_t ns = n - 8 * a.nvec;
    const unsigned grid = grid_for(a.nvec > ns ? a.nvec : ns, kCtasPerSmLight);
    const int w = store_width(gath + a.head);
#define ZERO_CAST_CASE(DT)                                                                      \
    switch (w) {                                                                                \
    case 16: launch_k(k_cast<DT, 16>, dim3(grid), dim3(kThreads), 0, s, a); break;              \
    case 8: launch_k(k_cast<DT, 8>, dim3(grid), dim3(kThreads), 0, s, a); break;                \
    case 4: launch_k(k_cast<DT, 4>, dim3(grid), dim3(kThreads), 0, s, a); break;                \
    default: launch_k(k_cast<DT, 2>, dim3(grid), dim3(kThreads), 0, s, a); break;               \
    }
    if (dtype == ZERO_F16) {
        ZERO_CAST_CASE(ZERO_F16)
    } else {
        ZERO_CAST_CASE(ZERO_BF16)
    }
#undef ZERO_CAST_CASE
}

bool loss_scale_valid(double ls) { return ls > 0.0 && ls <= 1.0e300; }

// [a, a + abytes) and [b, b + bbytes) share a byte (spans already checked
// not to wrap).
bool spans_overlap(const void* a, uint64_t abytes, const void* b, uint64_t bbytes)
{
    const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
    return x < y + bbytes && y < x + abytes;
}

}  // namespace

zero_status_t check_step_args(const zero_grads_t* g, const zero_layout_t* L,
                              const zero_state_t* in, const zero_state_t* out,
                              const void* gathered, uint64_t gathered_offset_elems,
                              uint64_t bucket_elems, double loss_scale, const zero_adamw_t* h,
                              const uint32_t* flag)
{
    if (!L || !gathered || !flag || bucket_elems == 0 || !loss_scale_valid(loss_scale) ||
        !adamw_valid(h))
        return ZERO_ERR_INVALID_ARG;
    if (L->nd == 0 || L->length > L->shard_elems)
        return ZERO_ERR_INVALID_ARG;
    const uint64_t n = L->length;
    zero_status_t st = check_grads(g, 0, n);
    if (st != ZERO_OK)
        return st;
    if (!aligned(gathered, 2) || !aligned(flag, 4))
        return ZERO_ERR_ALIGNMENT;
    st = check_state(in, out, n, 16);
    if (st != ZERO_OK)
        return st;
    // the gathered slot [gathered + offset, ... + n) must not wrap the
    // address space, and must share no byte with the state or the rows
    const uint64_t lim = 1ull << 61;
    if (gathered_offset_elems > lim || n > lim - gathered_offset_elems ||
        (uintptr_t)gathered > UINTPTR_MAX - 2 * (gathered_offset_elems + n))
        return ZERO_ERR_INVALID_ARG;
    const uint16_t* slot = static_cast<const uint16_t*>(gathered) + gathered_offset_elems;
    const float* st6[6] = {in->master, in->m, in->v, out->master, out->m, out->v};
    for (const float* p : st6)
        if (spans_overlap(slot, 2 * n, p, 4 * n))
            return ZERO_ERR_INVALID_ARG;
    const uint16_t* rows = static_cast<const uint16_t*>(g->base) + g->offset;
    const uint64_t row_span = (uint64_t)(g->nd - 1) * g->row_stride + n;
    if (n && spans_overlap(slot, 2 * n, rows, 2 * row_span))
        return ZERO_ERR_INVALID_ARG;
    return ZERO_OK;
}

namespace {

// Loads one fused-step kernel instance of `variant` now (asking CUDA for its
// attributes loads a lazily loaded kernel) and makes its shared-memory
// opt-in, so that launching it later calls nothing that could wait.
template <int DT, int W, bool V8>
void load_fused_w(int variant)
{
    cudaFuncAttributes fa;
    if (variant == 2) {
        (void)cudaFuncGetAttributes(&fa, k_step_fused_tma<DT, W, V8>);
        tma_opt_in<DT, W, V8>();
    } else if (variant == 1) {
        (void)cudaFuncGetAttributes(&fa, k_step_fused_ring<DT, W, V8, kModeStep>);
        ring_opt_in<DT, W, V8, kModeStep>();
    } else {
        (void)cudaFuncGetAttributes(&fa, k_step_fused<DT, W, V8>);
    }
}

template <int DT>
void load_fused_dt(int variant)
{
    if (variant == kVariantSmall || variant == kVariantAuto) {
        cudaFuncAttributes fa;
        (void)cudaFuncGetAttributes(&fa, k_step_fused_small<DT, 8, false>);
        (void)cudaFuncGetAttributes(&fa, k_step_fused_small<DT, 4, false>);
        (void)cudaFuncGetAttributes(&fa, k_step_fused_small<DT, 2, false>);
        (void)cudaFuncGetAttributes(&fa, k_step_fused_small<DT, 8, true>);
        (void)cudaFuncGetAttributes(&fa, k_step_fused_small<DT, 4, true>);
        (void)cudaFuncGetAttributes(&fa, k_step_fused_small<DT, 2, true>);
        if (variant == kVariantSmall)
            return;
        variant = 1;
    }
    load_fused_w<DT, 16, true>(variant);
    load_fused_w<DT, 8, true>(variant);
    load_fused_w<DT, 4, true>(variant);
    load_fused_w<DT, 2, true>(variant);
    load_fused_w<DT, 16, false>(variant);
    load_fused_w<DT, 8, false>(variant);
    load_fused_w<DT, 4, false>(variant);
    load_fused_w<DT, 2, false>(variant);
}

}  // namespace

bool pdl_launches() { return pdl_enabled(); }

void preload_fused(int dtype, bool host_rows)
{
    const int variant = fused_variant(host_rows);
    // per dtype and variant (kVariantAuto .. kVariantSmall): a bit per device
    static std::atomic<uint64_t> done[2][kVariantSmall - kVariantAuto + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        dev = 64;
    const uint64_t bit = dev < 64 ? 1ull << dev : 0;
    std::atomic<uint64_t>& d = done[dtype == ZERO_F16 ? 0 : 1][variant - kVariantAuto];
    if (bit && (d.load(std::memory_order_relaxed) & bit))
        return;
    if (dtype == ZERO_F16)
        load_fused_dt<ZERO_F16>(variant);
    else
        load_fused_dt<ZERO_BF16>(variant);
    (void)cudaGetLastError();
    if (bit)
        d.fetch_or(bit, std::memory_order_relaxed);
}

zero_status_t launch_fused_range(const uint16_t* rows, const zero_grads_t* g,
                                  const zero_state_t* in, const zero_state_t* out,
                                  uint16_t* gath, uint64_t b0, uint64_t len,
                                  const StepScalars& k, bool host_rows, uint32_t* d_nonfinite,
                                  const uint32_t* gate, void* stream)
{
    const int variant = fused_variant(host_rows);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const float* const sp[6] = {in->master, in->m, in->v, out->master, out->m, out->v};
    const bool v8 = state_v8_ok(sp);
    const uint64_t small_upto = variant == kVariantAuto ? small_window_limit() : 0;
    return for_each_window(elem_phase(rows + b0), len, kWindow, [&](uint64_t w0, uint64_t w1) {
        const uint64_t e0 = b0 + w0;
        FusedArgs a{rows + e0, g->row_stride, g->nd, split_window(g->offset + e0, w1 - w0),
                    in->master + e0, in->m + e0, in->v + e0, out->master + e0, out->m + e0,
                    out->v + e0, gath + e0, k, d_nonfinite, gate, nullptr,
                    (uint32_t)(w0 > 0)};
        const int v = variant != kVariantAuto ? variant
                                              : (w1 - w0 <= small_upto ? kVariantSmall : 1);
        if (v == kVariantSmall) {
            if (g->dtype == ZERO_F16)
                launch_small<ZERO_F16>(a, g->offset + e0, s);
            else
                launch_small<ZERO_BF16>(a, g->offset + e0, s);
            return launch_status();
        }
        const int width = store_width(gath + e0 + a.sp.head);
        if (g->dtype == ZERO_F16)
            launch_fused_dt<ZERO_F16>(a, width, v8, v, s);
        else
            launch_fused_dt<ZERO_BF16>(a, width, v8, v, s);
        return launch_status();
    });
}

}  // namespace zero

using namespace zero;

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

extern "C" zero_status_t zero_reduce_scatter_bucket(const zero_grads_t* g, uint64_t bucket_begin,
                                                    uint64_t bucket_len, float inv_scale,
                                                    float* cb_out, uint32_t* d_nonfinite,
                                                    void* stream)
{
    zero_status_t st = check_grads(g, bucket_begin, bucket_len);
    if (st != ZERO_OK)
        return st;
    if (!cb_out || !d_nonfinite)
        return ZERO_ERR_INVALID_ARG;
    if (!aligned(cb_out, 4) || !aligned(d_nonfinite, 4))
        return ZERO_ERR_ALIGNMENT;
    if (bucket_len == 0)
        return ZERO_OK;
    bool host_rows = false;
    zero_grads_t gr;   // the rows at the address the device reads them
    st = resolve_grads(g, &gr, &host_rows);
    if (st != ZERO_OK)
        return st;
    const void* words[2] = {cb_out, d_nonfinite};
    st = require_device(words, 2);
    if (st != ZERO_OK)
        return st;
    const int variant = fused_variant(host_rows);
    const uint16_t* first = static_cast<const uint16_t*>(gr.base) + g->offset + bucket_begin;
    return for_each_window(elem_phase(first), bucket_len, kWindow,
                           [&](uint64_t w0, uint64_t w1) {
        ReduceArgs a{first + w0, g->row_stride, g->nd,
                     split_window(g->offset + bucket_begin + w0, w1 - w0), inv_scale, cb_out + w0,
                     d_nonfinite, (uint32_t)(w0 > 0)};
        launch_reduce(a, g->dtype, variant, static_cast<cudaStream_t>(stream));
        return launch_status();
    });
}

extern "C" zero_status_t zero_check_nonfinite(const zero_grads_t* g, uint64_t begin, uint64_t n,
                                              uint32_t* d_nonfinite, void* stream)
{
    zero_status_t st = check_grads(g, begin, n);
    if (st != ZERO_OK)
        return st;
    if (!d_nonfinite)
        return ZERO_ERR_INVALID_ARG;
    if (!aligned(d_nonfinite, 4))
        return ZERO_ERR_ALIGNMENT;
    if (n == 0)
        return ZERO_OK;
    bool host_rows = false;
    zero_grads_t gr;   // the rows at the address the device reads them
    st = resolve_grads(g, &gr, &host_rows);
    if (st != ZERO_OK)
        return st;
    const void* word = d_nonfinite;
    st = require_device(&word, 1);
    if (st != ZERO_OK)
        return st;
    const int variant = fused_variant(host_rows);
    const uint16_t* first = static_cast<const uint16_t*>(gr.base) + g->offset + begin;
    return for_each_window(elem_phase(first), n, kWindow, [&](uint64_t w0, uint64_t w1) {
        ReduceArgs a{first + w0, g->row_stride, g->nd, split_window(g->offset + begin + w0, w1 - w0),
                     1.0f, nullptr, d_nonfinite, (uint32_t)(w0 > 0)};
        launch_reduce(a, g->dtype, variant, static_cast<cudaStream_t>(stream));
        return launch_status();
    });
}

extern "C" zero_status_t zero_adam_step_shard(const float* grad, const zero_state_t* in,
                                              const zero_state_t* out, uint64_t n,
                                              const zero_adamw_t* h, void* stream)
{
    if (!grad || !adamw_valid(h))
        return ZERO_ERR_INVALID_ARG;
    if (!aligned(grad, 4))
        return ZERO_ERR_ALIGNMENT;
    zero_status_t st = check_state(in, out, n, 4);
    if (st != ZERO_OK)
        return st;
    if (ranges_overlap(grad, out->master, n * 4) || ranges_overlap(grad, out->m, n * 4) ||
        ranges_overlap(grad, out->v, n * 4))
        return ZERO_ERR_INVALID_ARG;
    if (n == 0)
        return ZERO_OK;
    st = require_device_state(in, out, grad);
    if (st != ZERO_OK)
        return st;
    launch_adam(grad, in, out, n, make_scalars(h, 1, 1.0), static_cast<cudaStream_t>(stream));
    return launch_status();
}

extern "C" zero_status_t zero_gather_params_shard(const float* master, uint64_t n, void* gathered,
                                                  uint64_t slot_offset_elems, zero_dtype_t dtype,
                                                  void* stream)
{
    if (!master || !gathered || (dtype != ZERO_F16 && dtype != ZERO_BF16))
        return ZERO_ERR_INVALID_ARG;
    if (!aligned(master, 4) || !aligned(gathered, 2))
        return ZERO_ERR_ALIGNMENT;
    if (mul_overflows(n, 4) || slot_offset_elems > (UINT64_MAX >> 2))
        return ZERO_ERR_INVALID_ARG;
    if (n == 0)
        return ZERO_OK;
    if (ranges_overlap(static_cast<uint16_t*>(gathered) + slot_offset_elems, master, n * 4))
        return ZERO_ERR_INVALID_ARG;   // conservative: the larger extent
    void* gdev = nullptr;   // the slot at the address the device writes it
    zero_status_t st = resolve_ptr(gathered, &gdev);
    if (st != ZERO_OK)
        return st;
    const void* src = master;
    st = require_device(&src, 1);
    if (st != ZERO_OK)
        return st;
    uint16_t* slot = static_cast<uint16_t*>(gdev) + slot_offset_elems;
    launch_cast(master, n, slot, dtype, static_cast<cudaStream_t>(stream));
    return launch_status();
}

extern "C" zero_status_t zero_step_shard(const zero_grads_t* g, const zero_layout_t* L,
                                         const zero_state_t* in, const zero_state_t* out,
                                         void* gathered, uint64_t gathered_offset_elems,
                                         uint64_t bucket_elems, double loss_scale,
                                         const zero_adamw_t* h, uint32_t* d_nonfinite,
                                         void* stream)
{
    zero_status_t st = check_step_args(g, L, in, out, gathered, gathered_offset_elems,
                                       bucket_elems, loss_scale, h, d_nonfinite);
    if (st != ZERO_OK)
        return st;
    const uint64_t n = L->length;
    if (n == 0)
        return ZERO_OK;
    bool host_rows = false;
    zero_grads_t gr;   // the rows at the address the device reads them
    st = resolve_grads(g, &gr, &host_rows);
    if (st != ZERO_OK)
        return st;
    void* gdev = nullptr;   // the gathered buffer at the address the device writes it
    st = resolve_ptr(gathered, &gdev);
    if (st != ZERO_OK)
        return st;
    st = require_device_state(in, out, d_nonfinite);
    if (st != ZERO_OK)
        return st;
    const StepScalars k = make_scalars(h, g->nd, loss_scale);
    const uint16_t* rows = static_cast<const uint16_t*>(gr.base) + g->offset;
    uint16_t* gath = static_cast<uint16_t*>(gdev) + gathered_offset_elems;
    // The fused kernel keeps each reduced sum in registers, so a bucket is
    // never materialised and is no boundary of its work: the launch windows
    // are planned over the whole shard (one launch for shards of up to
    // kWindow elements, whatever the bucket size).
    return launch_fused_range(rows, g, in, out, gath, 0, n, k, host_rows, d_nonfinite, nullptr,
                               stream);
}

extern "C" zero_status_t zero_step_shard_unfused(const zero_grads_t* g, const zero_layout_t* L,
                                                 const zero_state_t* in, const zero_state_t* out,
                                                 void* gathered, uint64_t gathered_offset_elems,
                                                 uint64_t bucket_elems, double loss_scale,
                                                 const zero_adamw_t* h, float* cb,
                                                 uint64_t cb_elems, uint32_t* d_nonfinite,
                                                 void* stream)
{
    zero_status_t st = check_step_args(g, L, in, out, gathered, gathered_offset_elems,
                                       bucket_elems, loss_scale, h, d_nonfinite);
    if (st != ZERO_OK)
        return st;
    const uint64_t n = L->length;
    const uint64_t need = (bucket_elems < n ? bucket_elems : n) + 4;
    if (!cb || cb_elems < need)
        return ZERO_ERR_INVALID_ARG;
    if (!aligned(cb, 16))
        return ZERO_ERR_ALIGNMENT;
    if (n == 0)
        return ZERO_OK;
    bool host_rows = false;
    zero_grads_t gr;   // the rows at the address the device reads them
    st = resolve_grads(g, &gr, &host_rows);
    if (st != ZERO_OK)
        return st;
    void* gdev = nullptr;   // the gathered buffer at the address the device writes it
    st = resolve_ptr(gathered, &gdev);
    if (st != ZERO_OK)
        return st;
    st = require_device_state(in, out, d_nonfinite);
    if (st != ZERO_OK)
        return st;
    const void* workspace = cb;
    st = require_device(&workspace, 1);
    if (st != ZERO_OK)
        return st;
    const int variant = fused_variant(host_rows);
    const StepScalars k = make_scalars(h, g->nd, loss_scale);
    const StepScalars k_adam_only = make_scalars(h, 1, 1.0);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint16_t* rows = static_cast<const uint16_t*>(gr.base) + g->offset;
    uint16_t* gath = static_cast<uint16_t*>(gdev) + gathered_offset_elems;
    for (uint64_t b0 = 0; b0 < n; b0 += bucket_elems) {
        const uint64_t len = n - b0 < bucket_elems ? n - b0 : bucket_elems;
        // Shift the bucket inside cb so that cb and the state share a 16-byte
        // phase and the optimizer pass runs on float4s.
        float* cbb = cb + (b0 & 3);
        // the reduction in launch windows, like the fused step
        st = for_each_window(elem_phase(rows + b0), len, kWindow, [&](uint64_t w0, uint64_t w1) {
            ReduceArgs r{rows + b0 + w0, g->row_stride, g->nd,
                         split_window(g->offset + b0 + w0, w1 - w0), k.inv, cbb + w0,
                         d_nonfinite, (uint32_t)(w0 > 0)};
            launch_reduce(r, g->dtype, variant, s);
            return launch_status();
        });
        if (st != ZERO_OK)
            return st;
        const zero_state_t bin{in->master + b0, in->m + b0, in->v + b0};
        const zero_state_t bout{out->master + b0, out->m + b0, out->v + b0};
        launch_adam(cbb, &bin, &bout, len, k_adam_only, s);
        launch_cast(out->master + b0, len, gath + b0, g->dtype, s);
        st = launch_status();
        if (st != ZERO_OK)
            return st;
        if (len < bucket_elems)
            break;
    }
    return ZERO_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free unfused step: the fusion buffer lives in this library's own
// device memory instead of a caller-provided workspace.
// ---------------------------------------------------------------------------

namespace zero {
namespace {

// The fusion buffer: ZERO_STATIC_CB_ELEMS floats (16 MiB) on every device that
// loads the library.  In host code this name is only a stand-in for the
// symbol; kernels get the device address from cudaGetSymbolAddress.
__device__ __align__(256) float g_static_cb[ZERO_STATIC_CB_ELEMS];

// The id of the calling thread's current CUDA context (unique for the life of
// the process, never reused), or 0 if there is none or the driver cannot say.
// The two driver calls are found through the runtime, so the library still
// links no driver library; they only read the thread's context.
unsigned long long current_context_id()
{
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag found;
    std::call_once(found, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrent>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
        (void)cudaGetLastError();
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

constexpr int kMaxDevices = 128;
struct StaticCbEntry {
    unsigned long long ctx_id;   // context the address was looked up in (0: none yet)
    float* addr;
};
StaticCbEntry g_static_cb_addr[kMaxDevices];
std::mutex g_static_cb_mutex;

// Device address of g_static_cb on the current device.  It is looked up with
// cudaGetSymbolAddress (the device current) on the first call on a device and
// again whenever the device's context is not the one the address was found
// in (after cudaDeviceReset the library's device memory is loaded anew and
// the array may move); otherwise the cached address is returned.
zero_status_t static_cb_address(float** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return ZERO_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices)
        return ZERO_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_static_cb_mutex);
    StaticCbEntry& e = g_static_cb_addr[dev];
    const unsigned long long id = current_context_id();
    if (id == 0 || e.addr == nullptr || e.ctx_id != id) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_static_cb) != cudaSuccess || a == nullptr) {
            (void)cudaGetLastError();
            return ZERO_ERR_CUDA;
        }
        e.addr = static_cast<float*>(a);
        e.ctx_id = current_context_id();   // the lookup made the context current if it was not
    }
    *out = e.addr;
    return ZERO_OK;
}

}  // namespace
}  // namespace zero

extern "C" zero_status_t zero_step_shard_unfused_static(const zero_grads_t* g,
                                                        const zero_layout_t* L,
                                                        const zero_state_t* in,
                                                        const zero_state_t* out, void* gathered,
                                                        uint64_t gathered_offset_elems,
                                                        uint64_t bucket_elems, double loss_scale,
                                                        const zero_adamw_t* h,
                                                        uint32_t* d_nonfinite, void* stream)
{
    if (!L || bucket_elems == 0)
        return ZERO_ERR_INVALID_ARG;
    const uint64_t used = bucket_elems < L->length ? bucket_elems : L->length;
    if (used > ZERO_STATIC_CB_MAX_BUCKET)
        return ZERO_ERR_INVALID_ARG;   // the bucket does not fit the static fusion buffer
    zero_status_t st = check_step_args(g, L, in, out, gathered, gathered_offset_elems,
                                       bucket_elems, loss_scale, h, d_nonfinite);
    if (st != ZERO_OK)
        return st;
    float* cb = nullptr;
    st = static_cb_address(&cb);
    if (st != ZERO_OK)
        return st;
    return zero_step_shard_unfused(g, L, in, out, gathered, gathered_offset_elems, bucket_elems,
                                   loss_scale, h, cb, ZERO_STATIC_CB_ELEMS, d_nonfinite, stream);
}
