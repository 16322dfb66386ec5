// Host-only parts of the ZeRO shard-step C ABI: partition layout, model-state
// accounting, status strings and the fp32 step scalars.
//
// Partitioning follows "ZeRO: Memory Optimizations Toward Training Trillion
// Parameter Models", section "ZeRO-DP", Stage 1 (the state is split into Nd
// equal partitions and each rank owns one); the accounting follows section
// "Quantifying memory consumption" (2 + 2 + K bytes per parameter, K = 12) and
// the Stage 1-3 memory formulas of the same page.
#include <math.h>
#include <stdint.h>

#include "zero.h"
#include "zero_internal.h"

extern "C" const char* zero_status_string(zero_status_t status)
{
    switch (status) {
    case ZERO_OK: return "ZERO_OK";
    case ZERO_ERR_INVALID_ARG: return "ZERO_ERR_INVALID_ARG: invalid argument";
    case ZERO_ERR_ALIGNMENT: return "ZERO_ERR_ALIGNMENT: pointer or stride misaligned";
    case ZERO_ERR_CUDA: return "ZERO_ERR_CUDA: CUDA runtime error";
    case ZERO_ERR_TIMEOUT: return "ZERO_ERR_TIMEOUT: bounded wait expired";
    case ZERO_ERR_UNSUPPORTED: return "ZERO_ERR_UNSUPPORTED: not supported";
    case ZERO_ERR_IO: return "ZERO_ERR_IO: checkpoint file missing, unreadable or corrupt";
    }
    return "ZERO_ERR_UNKNOWN";
}

static uint64_t ceil_div(uint64_t a, uint64_t b) { return a / b + (a % b != 0); }

extern "C" zero_status_t zero_partition_layout(uint64_t psi, uint32_t nd, uint32_t rank,
                                               uint32_t row_align_elems, zero_layout_t* out)
{
    if (!out || nd == 0 || rank >= nd || row_align_elems == 0)
        return ZERO_ERR_INVALID_ARG;
    const uint64_t s = ceil_div(psi, nd);
    if (s != 0 && nd > UINT64_MAX / s)
        return ZERO_ERR_INVALID_ARG;
    const uint64_t pitch = ceil_div(s, row_align_elems) * row_align_elems;
    if (pitch < s)
        return ZERO_ERR_INVALID_ARG;
    const uint64_t begin = (uint64_t)rank * s;
    out->psi = psi;
    out->nd = nd;
    out->rank = rank;
    out->shard_elems = s;
    out->begin = begin;
    out->length = begin >= psi ? 0 : (psi - begin < s ? psi - begin : s);
    out->padded_elems = (uint64_t)nd * s;
    out->row_pitch = pitch;
    return ZERO_OK;
}

extern "C" uint64_t zero_model_state_bytes(uint64_t psi, uint32_t nd, uint32_t stage, uint32_t k)
{
    if (nd == 0 || stage > 3)
        return UINT64_MAX;
    const uint64_t bytes_per_param = 2 /* fp16 param */ + 2 /* fp16 grad */ + (uint64_t)k;
    if (psi != 0 && bytes_per_param > UINT64_MAX / psi)
        return UINT64_MAX;
    const uint64_t held = ceil_div(psi, nd);   // parameters of the partition a rank holds
    switch (stage) {
    case 0: return bytes_per_param * psi;                    // replicated everything
    case 1: return (2 + 2) * psi + (uint64_t)k * held;       // optimizer state partitioned
    case 2: return 2 * psi + (2 + (uint64_t)k) * held;       // + gradients partitioned
    default: return bytes_per_param * held;                  // + parameters partitioned
    }
}

extern "C" uint64_t zero_comm_volume_elems(uint64_t psi, uint32_t stage)
{
    if (stage > 3)
        return UINT64_MAX;
    const uint64_t times = stage == 3 ? 3 : 2;   // all-reduce (or RS + AG) 2, + param gathers 3
    if (psi > UINT64_MAX / times)
        return UINT64_MAX;
    return times * psi;
}

extern "C" uint64_t zero_model_state_bytes_mp(uint64_t psi, uint32_t nd, uint32_t nm,
                                              uint32_t stage, uint32_t k)
{
    if (nm == 0)
        return UINT64_MAX;
    return zero_model_state_bytes(ceil_div(psi, nm), nd, stage, k);   // one MP slice
}

namespace zero {

bool adamw_valid(const zero_adamw_t* h)
{
    if (!h || h->step == 0)
        return false;
    if (!(h->beta1 >= 0.0 && h->beta1 < 1.0) || !(h->beta2 >= 0.0 && h->beta2 < 1.0))
        return false;
    if (!isfinite(h->lr) || !isfinite(h->eps) || !isfinite(h->weight_decay))
        return false;
    return h->lr >= 0.0 && h->eps >= 0.0 && h->weight_decay >= 0.0;
}

StepScalars make_scalars(const zero_adamw_t* h, uint32_t nd, double loss_scale)
{
    const double t = (double)h->step;
    StepScalars k;
    k.inv = (float)(1.0 / ((double)nd * loss_scale));
    k.b1 = (float)h->beta1;
    k.b2 = (float)h->beta2;
    k.c1 = (float)(1.0 - h->beta1);
    k.c2 = (float)(1.0 - h->beta2);
    k.bc1 = (float)(1.0 - pow(h->beta1, t));
    k.bc2 = (float)(1.0 - pow(h->beta2, t));
    k.lr = (float)h->lr;
    k.eps = (float)h->eps;
    k.wdf = (float)(1.0 - h->lr * h->weight_decay);
    return k;
}

}  // namespace zero
