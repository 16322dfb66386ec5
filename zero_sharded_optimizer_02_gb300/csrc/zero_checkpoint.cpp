// Sharded checkpoints of the ZeRO optimizer state, with resharding.
//
// "ZeRO" (process-cxr ai-library), section on checkpointing and recovery: ZeRO
// training saves sharded checkpoints -- each rank writes only the state it
// owns -- which ties the checkpoint to the world size; whether a run can
// resume on a different number of GPUs and whether the metadata is stored
// reliably must be settled up front.
//
// One file per rank: a fixed header (format, partition, committed step,
// AdamW hyperparameters, a checksum of the payload) followed by the rank's
// fp32 master weights, m and v (length elements each).  Because ZeRO's step is
// elementwise over the flat parameter vector, resuming on a different Nd only
// moves elements: the loader fills the new rank's flat range from the
// overlapping ranges of the old files.  Host memory only; the caller moves
// state to and from the device.
#include <errno.h>
#include <stdio.h>
#include <string.h>

#include <string>
#include <thread>
#include <vector>

#include "zero.h"

namespace {

const char kMagic[8] = {'Z', 'E', 'R', 'O', 'C', 'K', 'P', 'T'};
constexpr uint32_t kVersion = 2;
constexpr uint64_t kFnvBasis = 0xCBF29CE484222325ull;
constexpr uint64_t kFnvPrime = 0x100000001B3ull;

// The payload checksum: 8 FNV-1a lanes over the payload's 32-bit words (word
// k to lane k mod 8), folded by FNV-1a over the lanes' bytes.  Every payload
// is a whole number of fp32 values and the lane follows the global word
// index, so the result does not depend on how the payload is split into
// chunks.
struct Fnv8 {
    uint64_t h[8] = {kFnvBasis, kFnvBasis, kFnvBasis, kFnvBasis,
                     kFnvBasis, kFnvBasis, kFnvBasis, kFnvBasis};
    uint64_t words = 0;

    void add(const void* p, size_t bytes)
    {
        const unsigned char* b = static_cast<const unsigned char*>(p);
        const size_t nw = bytes / 4;
        size_t i = 0;
        for (; i < nw && (words & 7); ++i, ++words)   // up to lane 0
            h[words & 7] = (h[words & 7] ^ word(b + 4 * i)) * kFnvPrime;
        uint64_t a0 = h[0], a1 = h[1], a2 = h[2], a3 = h[3];
        uint64_t a4 = h[4], a5 = h[5], a6 = h[6], a7 = h[7];
        for (; i + 8 <= nw; i += 8) {
            const unsigned char* q = b + 4 * i;
            a0 = (a0 ^ word(q)) * kFnvPrime;
            a1 = (a1 ^ word(q + 4)) * kFnvPrime;
            a2 = (a2 ^ word(q + 8)) * kFnvPrime;
            a3 = (a3 ^ word(q + 12)) * kFnvPrime;
            a4 = (a4 ^ word(q + 16)) * kFnvPrime;
            a5 = (a5 ^ word(q + 20)) * kFnvPrime;
            a6 = (a6 ^ word(q + 24)) * kFnvPrime;
            a7 = (a7 ^ word(q + 28)) * kFnvPrime;
            words += 8;
        }
        h[0] = a0, h[1] = a1, h[2] = a2, h[3] = a3;
        h[4] = a4, h[5] = a5, h[6] = a6, h[7] = a7;
        for (; i < nw; ++i, ++words)
            h[words & 7] = (h[words & 7] ^ word(b + 4 * i)) * kFnvPrime;
    }

    uint64_t value() const
    {
        uint64_t x = kFnvBasis;
        for (int l = 0; l < 8; ++l)
            for (int k = 0; k < 8; ++k)
                x = (x ^ ((h[l] >> (8 * k)) & 0xFF)) * kFnvPrime;
        return x;
    }

    static uint32_t word(const unsigned char* q)   // little-endian, any alignment
    {
        return (uint32_t)q[0] | (uint32_t)q[1] << 8 | (uint32_t)q[2] << 16 |
               (uint32_t)q[3] << 24;
    }
};

struct File {
    FILE* f = nullptr;
    ~File()
    {
        if (f)
            fclose(f);
    }
};

bool write_all(FILE* f, const void* p, size_t bytes)
{
    return fwrite(p, 1, bytes, f) == bytes;
}

bool read_all(FILE* f, void* p, size_t bytes)
{
    return fread(p, 1, bytes, f) == bytes;
}

zero_status_t read_header(FILE* f, zero_ckpt_header_t* h)
{
    if (!read_all(f, h, sizeof(*h)))
        return ZERO_ERR_IO;
    if (memcmp(h->magic, kMagic, 8) != 0 || h->version != kVersion ||
        h->header_bytes != sizeof(zero_ckpt_header_t))
        return ZERO_ERR_IO;
    zero_layout_t L;
    if (zero_partition_layout(h->psi, h->nd, h->rank, 1, &L) != ZERO_OK ||
        L.shard_elems != h->shard_elems || L.begin != h->begin || L.length != h->length)
        return ZERO_ERR_IO;
    return ZERO_OK;
}

// Streams the payload of an open file (positioned after the header) once:
// every chunk goes through the checksum, and the elements [r0, r1) of each of
// the three arrays are read straight into dst[a] + (element - r0).  Chunks
// are cut at r0 and r1, so a chunk lies wholly inside or wholly outside the
// range; those outside pass through a bounce buffer for the checksum alone.
// ZERO_ERR_IO on a short read or a checksum mismatch (dst is then
// unspecified).
zero_status_t load_payload(FILE* f, const zero_ckpt_header_t& h, uint64_t r0, uint64_t r1,
                           float* const dst[3])
{
    Fnv8 c;
    static const uint64_t kChunkElems = 1 << 20;
    std::vector<float> bounce;
    for (int a = 0; a < 3; ++a) {
        for (uint64_t e = 0; e < h.length;) {
            const uint64_t edge = e < r0 ? r0 : (e < r1 ? r1 : h.length);
            uint64_t take = edge - e < kChunkElems ? edge - e : kChunkElems;
            const bool inside = e >= r0 && e < r1;
            float* target;
            if (inside) {
                target = dst[a] + (e - r0);
            } else {
                if (bounce.empty())
                    bounce.resize(kChunkElems);
                target = bounce.data();
            }
            if (!read_all(f, target, (size_t)take * sizeof(float)))
                return ZERO_ERR_IO;
            c.add(target, (size_t)take * sizeof(float));
            e += take;
        }
    }
    return c.value() == h.payload_checksum ? ZERO_OK : ZERO_ERR_IO;
}

}  // namespace

extern "C" zero_status_t zero_checkpoint_save(const char* path, const zero_layout_t* L,
                                              const zero_adamw_t* h, const float* master,
                                              const float* m, const float* v)
{
    if (!path || !L || !h || (L->length && (!master || !m || !v)))
        return ZERO_ERR_INVALID_ARG;
    zero_layout_t chk;
    if (zero_partition_layout(L->psi, L->nd, L->rank, 1, &chk) != ZERO_OK ||
        chk.length != L->length || chk.begin != L->begin)
        return ZERO_ERR_INVALID_ARG;
    zero_ckpt_header_t hd;
    memset(&hd, 0, sizeof(hd));
    memcpy(hd.magic, kMagic, 8);
    hd.version = kVersion;
    hd.header_bytes = sizeof(hd);
    hd.psi = L->psi;
    hd.nd = L->nd;
    hd.rank = L->rank;
    hd.shard_elems = chk.shard_elems;
    hd.begin = chk.begin;
    hd.length = chk.length;
    hd.step = h->step;
    hd.lr = h->lr;
    hd.beta1 = h->beta1;
    hd.beta2 = h->beta2;
    hd.eps = h->eps;
    hd.weight_decay = h->weight_decay;
    // The checksum runs on a second thread over the in-memory arrays while
    // this one writes them; the header, written first with a zero checksum,
    // is rewritten at the end.  The file is written under a temporary name
    // and renamed, so a crash never leaves a torn file at `path`.
    const size_t bytes = (size_t)L->length * sizeof(float);
    const float* arrays[3] = {master, m, v};
    uint64_t sum = 0;
    auto checksum = [&]() {
        Fnv8 c;
        for (const float* a : arrays)
            c.add(a, bytes);
        sum = c.value();
    };
    std::thread worker;
    try {
        worker = std::thread(checksum);
    } catch (...) {   // no thread to be had: sum inline after the writes
    }
    const std::string tmp = std::string(path) + ".tmp";
    bool ok;
    {
        File f;
        f.f = fopen(tmp.c_str(), "wb");
        ok = f.f != nullptr && write_all(f.f, &hd, sizeof(hd));
        for (int a = 0; a < 3 && ok; ++a)
            ok = write_all(f.f, arrays[a], bytes);
        if (worker.joinable())
            worker.join();
        else
            checksum();
        hd.payload_checksum = sum;
        ok = ok && fseeko(f.f, 0, SEEK_SET) == 0 && write_all(f.f, &hd, sizeof(hd)) &&
             fflush(f.f) == 0;
    }
    if (!ok) {
        remove(tmp.c_str());
        return ZERO_ERR_IO;
    }
    if (rename(tmp.c_str(), path) != 0) {
        remove(tmp.c_str());
        return ZERO_ERR_IO;
    }
    return ZERO_OK;
}

extern "C" zero_status_t zero_checkpoint_read_header(const char* path, zero_ckpt_header_t* out)
{
    if (!path || !out)
        return ZERO_ERR_INVALID_ARG;
    File f;
    f.f = fopen(path, "rb");
    if (!f.f)
        return ZERO_ERR_IO;
    return read_header(f.f, out);
}

extern "C" zero_status_t zero_checkpoint_load(const char* const* paths, uint32_t n_paths,
                                              const zero_layout_t* L, float* master, float* m,
                                              float* v, zero_adamw_t* h_out)
{
    if (!paths || n_paths == 0 || !L || (L->length && (!master || !m || !v)))
        return ZERO_ERR_INVALID_ARG;
    zero_layout_t Ln;
    if (zero_partition_layout(L->psi, L->nd, L->rank, 1, &Ln) != ZERO_OK ||
        Ln.length != L->length || Ln.begin != L->begin)
        return ZERO_ERR_INVALID_ARG;
    // headers of every old rank: same partition, same step, rank r in paths[r]
    zero_ckpt_header_t first;
    memset(&first, 0, sizeof(first));
    for (uint32_t r = 0; r < n_paths; ++r) {
        if (!paths[r])
            return ZERO_ERR_INVALID_ARG;
        zero_ckpt_header_t hd;
        zero_status_t st = zero_checkpoint_read_header(paths[r], &hd);
        if (st != ZERO_OK)
            return st;
        if (hd.nd != n_paths || hd.rank != r || hd.psi != L->psi)
            return ZERO_ERR_INVALID_ARG;
        if (r == 0)
            first = hd;
        else if (hd.step != first.step)
            return ZERO_ERR_IO;
    }
    const uint64_t s_old = first.shard_elems;
    const uint64_t lo_new = Ln.begin, hi_new = Ln.begin + Ln.length;
    float* dst[3] = {master, m, v};
    for (uint32_t r = 0; r < n_paths && Ln.length; ++r) {
        const uint64_t lo_old = (uint64_t)r * s_old;
        zero_ckpt_header_t hd;
        File f;
        f.f = fopen(paths[r], "rb");
        if (!f.f || read_header(f.f, &hd) != ZERO_OK)
            return ZERO_ERR_IO;
        const uint64_t hi_old = lo_old + hd.length;
        const uint64_t lo = lo_old > lo_new ? lo_old : lo_new;
        const uint64_t hi = hi_old < hi_new ? hi_old : hi_new;
        if (lo >= hi)
            continue;
        // one pass over the file: checked whole, its part of the new range read
        // into place
        float* const at[3] = {dst[0] + (lo - lo_new), dst[1] + (lo - lo_new),
                              dst[2] + (lo - lo_new)};
        const zero_status_t st = load_payload(f.f, hd, lo - lo_old, hi - lo_old, at);
        if (st != ZERO_OK)
            return st;
    }
    if (h_out) {
        h_out->lr = first.lr;
        h_out->beta1 = first.beta1;
        h_out->beta2 = first.beta2;
        h_out->eps = first.eps;
        h_out->weight_decay = first.weight_decay;
        h_out->step = first.step;
    }
    return ZERO_OK;
}
