// ZeRO-3 on-demand gather of a flat parameter range (sm_103a).
//
// "ZeRO: Memory Optimizations Toward Training Trillion Parameter Models",
// section "ZeRO-DP", Stage 3: parameters are partitioned too; before a layer
// runs, its parameters are collected from the ranks that own them and
// released after use.  With Nd ranks emulated in one GPU's memory, the
// collection of a layer's flat range [begin, begin + len) is a copy of at most
// ceil(len / S) + 1 contiguous shard segments into a contiguous buffer.  The
// same copy, on 4-byte elements, moves fp32 optimizer state between shard
// layouts (resharding to another Nd).
//
// Up to 48 segments go into one launch (the plans ride in the kernel
// parameters); each CTA copies a contiguous run of one segment.  A segment's body is copied in 16-byte destination chunks:
// when source and destination differ in 16-byte phase by DELTA bytes, each
// chunk is assembled from two aligned 16-byte source loads with funnel
// shifts, so every global access stays a full 16-byte vector.  Elements at
// the two ends whose aligned source chunks would extend past the segment are
// copied one 2-byte unit at a time, so nothing outside the segment is read.
#include <cuda_runtime.h>
#include <stdint.h>

#include "zero.h"
#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kCopyThreads = 256;

// One contiguous copy of a segment, planned on the host (see plan_segment).
struct SegCopy {
    const uint16_t* src;   // segment start (2-byte aligned)
    uint16_t* dst;         // destination start (2-byte aligned)
    const uint4* a;        // aligned source chunk feeding body chunk 0
    uint4* d;              // body chunk 0 (16-byte aligned)
    uint32_t delta;        // source-destination phase difference in bytes (even, < 16)
    uint32_t pad;
    uint64_t units;        // 2-byte units in the segment
    uint64_t nchunks;      // 16-byte destination chunks in the body
    uint64_t body_lo;      // first unit of the body
};

// Up to kMaxSegs segments per launch, passed by value in the kernel
// parameters.  Every CTA copies one contiguous run of kChunksPerCta body
// chunks of one segment (block_end is the inclusive prefix sum of the CTAs
// each segment gets); a segment's first CTA also copies its edge units.
constexpr int kMaxSegs = (int)ZERO_GATHER_SEGMENTS_PER_LAUNCH;
constexpr int kChunksPerThread = 8;
constexpr uint64_t kChunksPerCta = (uint64_t)kCopyThreads * kChunksPerThread;

struct SegBatch {
    int nseg;
    SegCopy seg[kMaxSegs];
    uint64_t block_end[kMaxSegs];
};

// Bytes [DELTA, DELTA + 16) of the 32-byte window x:y (DELTA even, 0..14).
template <int DELTA>
__device__ __forceinline__ uint4 window16(const uint4& x, const uint4& y)
{
    const uint32_t w[8] = {x.x, x.y, x.z, x.w, y.x, y.y, y.z, y.w};
    constexpr int q = DELTA / 4;
    constexpr int r = (DELTA % 4) * 8;   // 0 or 16 bits
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        o[i] = r == 0 ? w[i + q] : __funnelshift_r(w[i + q], w[i + q + 1], r);
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Copies body chunks [k0, k1) of segment c, kChunksPerThread per thread.
template <int DELTA>
__device__ __forceinline__ void copy_chunks(const SegCopy& c, uint64_t k0, uint64_t k1)
{
    uint4 x[kChunksPerThread], y[kChunksPerThread];
#pragma unroll
    for (int i = 0; i < kChunksPerThread; ++i) {
        const uint64_t k = k0 + (uint64_t)i * kCopyThreads + threadIdx.x;
        if (k < k1) {
            x[i] = __ldcs(c.a + k);
            y[i] = DELTA ? __ldcs(c.a + k + 1) : x[i];
        }
    }
#pragma unroll
    for (int i = 0; i < kChunksPerThread; ++i) {
        const uint64_t k = k0 + (uint64_t)i * kCopyThreads + threadIdx.x;
        if (k < k1)
            __stcs(c.d + k, window16<DELTA>(x[i], y[i]));
    }
}

__global__ void __launch_bounds__(kCopyThreads) k_gather_segments(const SegBatch b)
{
    __shared__ int s_seg;
    if (threadIdx.x == 0) {   // the segment this CTA belongs to
        int lo = 0, hi = b.nseg - 1;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (b.block_end[mid] > blockIdx.x)
                hi = mid;
            else
                lo = mid + 1;
        }
        s_seg = lo;
    }
    __syncthreads();
    const int si = s_seg;
    const SegCopy c = b.seg[si];
    const uint64_t local_block = blockIdx.x - (si ? b.block_end[si - 1] : 0);
    if (local_block == 0) {   // edge units of the segment, 2 bytes each
        const uint64_t body_hi = c.body_lo + 8 * c.nchunks;
        const uint64_t nedge = c.units - 8 * c.nchunks;
        for (uint64_t t = threadIdx.x; t < nedge; t += kCopyThreads) {
            const uint64_t u = t < c.body_lo ? t : body_hi + (t - c.body_lo);
            c.dst[u] = c.src[u];
        }
    }
    const uint64_t k0 = local_block * kChunksPerCta;
    const uint64_t k1 = k0 + kChunksPerCta < c.nchunks ? k0 + kChunksPerCta : c.nchunks;
    if (k0 >= k1)
        return;
    switch (c.delta) {        // uniform within the CTA
    case 0: copy_chunks<0>(c, k0, k1); break;
    case 2: copy_chunks<2>(c, k0, k1); break;
    case 4: copy_chunks<4>(c, k0, k1); break;
    case 6: copy_chunks<6>(c, k0, k1); break;
    case 8: copy_chunks<8>(c, k0, k1); break;
    case 10: copy_chunks<10>(c, k0, k1); break;
    case 12: copy_chunks<12>(c, k0, k1); break;
    default: copy_chunks<14>(c, k0, k1); break;
    }
}

// Plans the copy of `units` 2-byte units from src to dst: a 16-byte chunk
// body whose source chunks lie inside the segment, and edge units.
SegCopy plan_segment(const uint16_t* src, uint16_t* dst, uint64_t units)
{
    SegCopy c{src, dst, nullptr, nullptr, 0, 0, units, 0, units};
    const uintptr_t S = (uintptr_t)src, D = (uintptr_t)dst;
    const uint64_t nbytes = 2 * units;
    const uint64_t dpre = (16 - (D & 15)) & 15;          // bytes before dst is aligned
    if (nbytes >= 64 + dpre) {
        const uintptr_t S1 = S + dpre;                    // source byte of dst chunk 0
        const uint32_t delta = (uint32_t)(S1 & 15);
        const uintptr_t A = S1 - delta;                   // aligned source chunk of dst chunk 0
        // dst chunk k reads source chunks A+16k and (delta > 0) A+16(k+1); both
        // must lie inside [S, S + nbytes).
        const uint64_t k0 = A < S ? 1 : 0;
        const uint64_t src_chunks = (S + nbytes - A) / 16;        // whole chunks from A
        const uint64_t k_end_src = src_chunks >= (delta ? 2u : 1u) ? src_chunks - (delta ? 1 : 0) : 0;
        const uint64_t k_end_dst = (nbytes - dpre) / 16;
        const uint64_t k1 = k_end_src < k_end_dst ? k_end_src : k_end_dst;
        if (k1 > k0) {
            c.a = reinterpret_cast<const uint4*>(A) + k0;
            c.d = reinterpret_cast<uint4*>(D + dpre) + k0;
            c.delta = delta;
            c.nchunks = k1 - k0;
            c.body_lo = (dpre + 16 * k0) / 2;
        }
    }
    return c;
}

zero_status_t launch_batch(SegBatch& b, cudaStream_t s)
{
    if (b.nseg == 0)
        return ZERO_OK;
    uint64_t blocks = 0;
    for (int i = 0; i < b.nseg; ++i) {
        const uint64_t nb = (b.seg[i].nchunks + kChunksPerCta - 1) / kChunksPerCta;
        blocks += nb ? nb : 1;                 // at least one CTA: the edge units
        b.block_end[i] = blocks;
    }
    if (blocks > 0x7FFFFFFFull)
        return ZERO_ERR_INVALID_ARG;
    k_gather_segments<<<(unsigned)blocks, kCopyThreads, 0, s>>>(b);
    b.nseg = 0;
    return cudaGetLastError() == cudaSuccess ? ZERO_OK : ZERO_ERR_CUDA;
}

}  // namespace
}  // namespace zero

extern "C" zero_status_t zero_gather_range(const void* shards, uint64_t pitch, uint64_t psi,
                                           uint32_t nd, uint64_t begin, uint64_t len,
                                           uint32_t elem_bytes, void* out, void* stream)
{
    if (!shards || !out || nd == 0 || (elem_bytes != 2 && elem_bytes != 4))
        return ZERO_ERR_INVALID_ARG;
    if (begin > psi || len > psi - begin)
        return ZERO_ERR_INVALID_ARG;
    const uint64_t s = psi / nd + (psi % nd != 0);
    if (pitch < s || (nd > 1 && pitch > (UINT64_MAX / 8) / nd))
        return ZERO_ERR_INVALID_ARG;
    if (((uintptr_t)shards & (elem_bytes - 1)) || ((uintptr_t)out & (elem_bytes - 1)))
        return ZERO_ERR_ALIGNMENT;
    const uintptr_t sb = (uintptr_t)shards, se = sb + (uint64_t)nd * pitch * elem_bytes;
    const uintptr_t ob = (uintptr_t)out, oe = ob + len * elem_bytes;
    if (len && ob < se && sb < oe)
        return ZERO_ERR_INVALID_ARG;   // out overlaps the shards
    if (len == 0)
        return ZERO_OK;
    // where the kernel reads and writes: device or managed memory as is,
    // page-locked host memory at its device mapping; anything else (pageable
    // host memory) is refused before anything is launched
    void* sdev = nullptr;
    void* odev = nullptr;
    zero_status_t rs = zero::resolve_ptr(shards, &sdev);
    if (rs != ZERO_OK)
        return rs;
    rs = zero::resolve_ptr(out, &odev);
    if (rs != ZERO_OK)
        return rs;
    shards = sdev;
    out = odev;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint64_t units_per_elem = elem_bytes / 2;
    zero::SegBatch batch;
    batch.nseg = 0;
    uint64_t done = 0;
    while (done < len) {
        const uint64_t flat = begin + done;
        const uint64_t r = flat / s, local = flat % s;
        const uint64_t take = (s - local) < (len - done) ? (s - local) : (len - done);
        const uint16_t* src = static_cast<const uint16_t*>(shards) +
                              (r * pitch + local) * units_per_elem;
        uint16_t* dst = static_cast<uint16_t*>(out) + done * units_per_elem;
        batch.seg[batch.nseg++] = zero::plan_segment(src, dst, take * units_per_elem);
        if (batch.nseg == zero::kMaxSegs) {
            const zero_status_t r2 = zero::launch_batch(batch, st);
            if (r2 != ZERO_OK)
                return r2;
        }
        done += take;
    }
    const zero_status_t r3 = zero::launch_batch(batch, st);
    if (r3 != ZERO_OK)
        return r3;
    return ZERO_OK;
}
