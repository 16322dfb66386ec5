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
// Each segment is one launch.  Its body is copied in 16-byte destination
// chunks: when source and destination differ in 16-byte phase by DELTA bytes,
// each chunk is assembled from two aligned 16-byte source loads with funnel
// shifts, so every global access stays a full 16-byte vector.  Elements at
// the two ends whose aligned source chunks would extend past the segment are
// copied one 2-byte unit at a time, so nothing outside the segment is read.
#include <cuda_runtime.h>
#include <stdint.h>

#include "zero.h"

namespace zero {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyCtasPerSm = 8;

struct SegCopy {
    const uint16_t* src;   // segment start (2-byte aligned)
    uint16_t* dst;         // destination start (2-byte aligned)
    uint64_t units;        // 2-byte units in the segment
    const uint4* a;        // aligned source chunk feeding destination chunk k0
    uint4* d;              // destination chunk k0 (16-byte aligned)
    uint64_t nchunks;      // 16-byte destination chunks in the body
    uint64_t body_lo;      // first unit of the body
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

template <int DELTA>
__global__ void __launch_bounds__(kCopyThreads, kCopyCtasPerSm) k_gather_segment(const SegCopy c)
{
    const uint64_t tid = (uint64_t)blockIdx.x * kCopyThreads + threadIdx.x;
    const uint64_t nthr = (uint64_t)gridDim.x * kCopyThreads;
    // edges: units before the body and after it
    const uint64_t body_hi = c.body_lo + 8 * c.nchunks;
    const uint64_t edge = c.body_lo + (c.units - body_hi);
    for (uint64_t t = tid; t < edge; t += nthr) {
        const uint64_t u = t < c.body_lo ? t : body_hi + (t - c.body_lo);
        c.dst[u] = c.src[u];
    }
    for (uint64_t k = tid; k < c.nchunks; k += nthr) {
        const uint4 x = __ldcs(c.a + k);
        const uint4 y = DELTA ? __ldcs(c.a + k + 1) : x;
        __stcs(c.d + k, window16<DELTA>(x, y));
    }
}

int sm_count_gather()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms <= 0)
        sms = 1;
    return sms;
}

// Plans and launches the copy of `units` 2-byte units from src to dst.
void copy_segment(const uint16_t* src, uint16_t* dst, uint64_t units, cudaStream_t s)
{
    SegCopy c{src, dst, units, nullptr, nullptr, 0, units};
    const uintptr_t S = (uintptr_t)src, D = (uintptr_t)dst;
    const uint64_t nbytes = 2 * units;
    const uint64_t dpre = (16 - (D & 15)) & 15;          // bytes before dst is aligned
    int delta = 0;
    if (nbytes >= 64 + dpre) {
        const uintptr_t S1 = S + dpre;                    // source byte of dst chunk 0
        delta = (int)(S1 & 15);
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
            c.nchunks = k1 - k0;
            c.body_lo = (dpre + 16 * k0) / 2;
        }
    }
    const uint64_t work = c.nchunks > 64 ? c.nchunks : 64;
    uint64_t grid = (work + kCopyThreads - 1) / kCopyThreads;
    const uint64_t cap = (uint64_t)sm_count_gather() * kCopyCtasPerSm;
    grid = grid < cap ? grid : cap;
    switch (delta) {
    case 0: k_gather_segment<0><<<(unsigned)grid, kCopyThreads, 0, s>>>(c); break;
    case 2: k_gather_segment<2><<<(unsigned)grid, kCopyThreads, 0, s>>>(c); break;
    case 4: k_gather_segment<4><<<(unsigned)grid, kCopyThreads, 0, s>>>(c); break;
    case 6: k_gather_segment<6><<<(unsigned)grid, kCopyThreads, 0, s>>>(c); break;
    case 8: k_gather_segment<8><<<(unsigned)grid, kCopyThreads, 0, s>>>(c); break;
    case 10: k_gather_segment<10><<<(unsigned)grid, kCopyThreads, 0, s>>>(c); break;
    case 12: k_gather_segment<12><<<(unsigned)grid, kCopyThreads, 0, s>>>(c); break;
    default: k_gather_segment<14><<<(unsigned)grid, kCopyThreads, 0, s>>>(c); break;
    }
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
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint64_t units_per_elem = elem_bytes / 2;
    uint64_t done = 0;
    while (done < len) {
        const uint64_t flat = begin + done;
        const uint64_t r = flat / s, local = flat % s;
        const uint64_t take = (s - local) < (len - done) ? (s - local) : (len - done);
        const uint16_t* src = static_cast<const uint16_t*>(shards) +
                              (r * pitch + local) * units_per_elem;
        uint16_t* dst = static_cast<uint16_t*>(out) + done * units_per_elem;
        zero::copy_segment(src, dst, take * units_per_elem, st);
        if (cudaGetLastError() != cudaSuccess)
            return ZERO_ERR_CUDA;
        done += take;
    }
    return ZERO_OK;
}
