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

#include "zero.h"

namespace {

const char kMagic[8] = {'Z', 'E', 'R', 'O', 'C', 'K', 'P', 'T'};

// FNV-1a (64-bit state) over the payload's 32-bit words.  Every payload is a
// whole number of fp32 values, so the result does not depend on how the
// payload is split into chunks.
struct Fnv {
    uint64_t h = 0xCBF29CE484222325ull;
    void add(const void* p, size_t bytes)
    {
        const unsigned char* b = static_cast<const unsigned char*>(p);
        for (size_t i = 0; i + 4 <= bytes; i += 4) {
            uint32_t w;
            memcpy(&w, b + i, 4);
            h = (h ^ w) * 0x100000001B3ull;
        }
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
    if (memcmp(h->magic, kMagic, 8) != 0 || h->version != 1 ||
        h->header_bytes != sizeof(zero_ckpt_header_t))
        return ZERO_ERR_IO;
    zero_layout_t L;
    if (zero_partition_layout(h->psi, h->nd, h->rank, 1, &L) != ZERO_OK ||
        L.shard_elems != h->shard_elems || L.begin != h->begin || L.length != h->length)
        return ZERO_ERR_IO;
    return ZERO_OK;
}

// Streams the payload of an open file (positioned after the header) through
// the checksum and compares.
zero_status_t verify_payload(FILE* f, const zero_ckpt_header_t& h)
{
    Fnv c;
    static const size_t kChunk = 1 << 22;
    std::string buf(kChunk, '\0');
    uint64_t left = 3 * h.length * sizeof(float);
    while (left) {
        const size_t take = left < kChunk ? (size_t)left : kChunk;
        if (!read_all(f, &buf[0], take))
            return ZERO_ERR_IO;
        c.add(buf.data(), take);
        left -= take;
    }
    return c.h == h.payload_checksum ? ZERO_OK : ZERO_ERR_IO;
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
    hd.version = 1;
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
    const size_t bytes = (size_t)L->length * sizeof(float);
    Fnv c;
    c.add(master, bytes);
    c.add(m, bytes);
    c.add(v, bytes);
    hd.payload_checksum = c.h;
    // write to a temporary name, then rename: a crash never leaves a torn file
    const std::string tmp = std::string(path) + ".tmp";
    {
        File f;
        f.f = fopen(tmp.c_str(), "wb");
        if (!f.f)
            return ZERO_ERR_IO;
        if (!write_all(f.f, &hd, sizeof(hd)) || !write_all(f.f, master, bytes) ||
            !write_all(f.f, m, bytes) || !write_all(f.f, v, bytes) || fflush(f.f) != 0) {
            remove(tmp.c_str());
            return ZERO_ERR_IO;
        }
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
        zero_status_t st = verify_payload(f.f, hd);   // every file read is checked whole
        if (st != ZERO_OK)
            return st;
        for (int a = 0; a < 3; ++a) {
            const long long off = (long long)sizeof(hd) +
                                  (long long)((a * hd.length + (lo - lo_old)) * sizeof(float));
            if (fseeko(f.f, off, SEEK_SET) != 0 ||
                !read_all(f.f, dst[a] + (lo - lo_new), (size_t)(hi - lo) * sizeof(float)))
                return ZERO_ERR_IO;
        }
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
