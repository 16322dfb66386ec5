/*
 * CPU oracle of the ZeRO partitioned optimizer step -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct restatement of what one data-parallel rank
 * computes in ZeRO's optimizer step.  Only the tests, the package's smoke check
 * and the benchmark's CPU-baseline leg load this file's library; the CUDA
 * library never links, includes or calls it, and the two share no code.
 *
 * What the sources fix (page title, section):
 *   - "ZeRO: Memory Optimizations Toward Training Trillion Parameter Models"
 *     (notes.yuuk.io summary), section "Quantifying memory consumption":
 *     mixed-precision Adam keeps fp16 parameters and gradients and fp32
 *     master weights, momentum and variance: 2+2+4+4+4 = 16 bytes per
 *     parameter, K = 12 the optimizer-state multiplier.
 *   - Same page, "ZeRO-DP" Stages 1-3: the state is split into Nd equal
 *     partitions, each rank updates only its 1/Nd, gradients are
 *     reduce-scattered bucket by bucket, parameters all-gathered at the end of
 *     the step; the per-rank memory formulas and the 7.5B-parameter table.
 *   - Same page, "ZeRO-R / CB": a constant-size fusion buffer.
 *   - "ZeRO" (process-cxr ai-library), sections on memory background and the
 *     M_DDP / M_ZeRO-1/2/3 formulas.
 * What the sources leave open and the readings taken here:
 *   - The Adam(W) update: Adam (Kingma & Ba, ICLR 2015) with bias correction
 *     and eps outside the square root, plus decoupled weight decay
 *     (Loshchilov & Hutter, ICLR 2019) applied as p * (1 - lr * wd).
 *   - Reduction order: a sequential left fold over ranks 0..Nd-1 in fp32.
 *   - Scaling: one fp32 multiply of the sum by fp32(1 / (Nd * loss_scale)).
 *   - Skip: any nonfinite reduced sum skips the step on every shard.
 *   - Scalars are formed in fp64 and rounded once to fp32.
 *   - Accounting with a padded last shard counts S = ceil(Psi / Nd) per rank.
 * Precision: the pages fix fp32 for master weights and moments and fp16 for
 * parameters and gradients, so the step is computed in fp32 with every
 * operation correctly rounded (built with -ffp-contract=off); an fp64 shadow
 * of the same formulas is provided to bound the fp32 result.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#define ORC_F16 0
#define ORC_BF16 1

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 and bfloat16, written from their definitions.          */
/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits.                */
/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits.                */
/* ------------------------------------------------------------------------ */

typedef struct {
    int frac_bits;  /* stored fraction bits */
    int bias;       /* exponent bias */
    int emin;       /* exponent of the smallest normal binade */
    int emax;       /* exponent of the largest finite binade */
    int exp_all1;   /* exponent field of inf/NaN */
} orc_fmt_t;

static const orc_fmt_t FMT_F16 = {10, 15, -14, 15, 0x1f};
static const orc_fmt_t FMT_BF16 = {7, 127, -126, 127, 0xff};

static float decode16(uint16_t h, const orc_fmt_t* f)
{
    int sign = h >> 15;
    int e = (h >> f->frac_bits) & f->exp_all1;
    int frac = h & ((1 << f->frac_bits) - 1);
    double mag;
    if (e == f->exp_all1) {
        if (frac)
            return sign ? -NAN : NAN;
        return sign ? -INFINITY : INFINITY;
    }
    if (e == 0) /* subnormal: frac * 2^(emin - frac_bits) */
        mag = ldexp((double)frac, f->emin - f->frac_bits);
    else /* normal: (1.frac) * 2^(e - bias) */
        mag = ldexp((double)(frac | (1 << f->frac_bits)), e - f->bias - f->frac_bits);
    return (float)(sign ? -mag : mag); /* exact: fp32 holds every value */
}

/* Round-to-nearest-even encoding of a float into the 16-bit format. */
static uint16_t encode16(float x, const orc_fmt_t* f)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    uint16_t inf = (uint16_t)(f->exp_all1 << f->frac_bits);
    if (isnan(x))
        return sign | inf | (uint16_t)(1 << (f->frac_bits - 1));
    if (isinf(x))
        return sign | inf;
    double ax = fabs((double)x);
    if (ax == 0.0)
        return sign;
    int e2;
    frexp(ax, &e2);            /* ax = mant * 2^e2, mant in [0.5, 1) */
    int E = e2 - 1;            /* floor(log2(ax)) */
    if (E < f->emin)
        E = f->emin;           /* subnormals share the smallest binade's spacing */
    double quantum = ldexp(1.0, E - f->frac_bits);
    double r = nearbyint(ax / quantum) * quantum; /* ties to even; exact */
    if (r >= ldexp(1.0, f->emax + 1))
        return sign | inf;     /* rounded past the largest finite value */
    if (r == 0.0)
        return sign;
    frexp(r, &e2);
    E = e2 - 1;
    if (E < f->emin) /* subnormal result */
        return sign | (uint16_t)(r / ldexp(1.0, f->emin - f->frac_bits));
    uint32_t frac = (uint32_t)(r / ldexp(1.0, E - f->frac_bits)) - (1u << f->frac_bits);
    uint32_t biased = (uint32_t)(E + f->bias);
    return sign | (uint16_t)((biased << f->frac_bits) | frac);
}

float orc_half_to_float(uint16_t h) { return decode16(h, &FMT_F16); }
float orc_bf16_to_float(uint16_t h) { return decode16(h, &FMT_BF16); }
uint16_t orc_float_to_half(float x) { return encode16(x, &FMT_F16); }
uint16_t orc_float_to_bf16(float x) { return encode16(x, &FMT_BF16); }

void orc_decode_n(const uint16_t* in, float* out, uint64_t n, int dtype)
{
    for (uint64_t i = 0; i < n; ++i)
        out[i] = dtype == ORC_F16 ? orc_half_to_float(in[i]) : orc_bf16_to_float(in[i]);
}

void orc_encode_n(const float* in, uint16_t* out, uint64_t n, int dtype)
{
    for (uint64_t i = 0; i < n; ++i)
        out[i] = dtype == ORC_F16 ? orc_float_to_half(in[i]) : orc_float_to_bf16(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Partitioning and memory accounting (ZeRO-DP, Stages 1-3).                 */
/* ------------------------------------------------------------------------ */

/* Equal partition of Psi over Nd ranks with a zero-padded last shard:
 * out = {S = ceil(Psi/Nd), begin = rank*S, n = max(0, min(S, Psi - begin))}. */
int orc_layout(uint64_t psi, uint32_t nd, uint32_t rank, uint64_t out[3])
{
    if (nd == 0 || rank >= nd)
        return -1;
    uint64_t s = psi / nd + (psi % nd != 0);
    uint64_t begin = (uint64_t)rank * s;
    uint64_t n = 0;
    if (begin < psi)
        n = psi - begin < s ? psi - begin : s;
    out[0] = s;
    out[1] = begin;
    out[2] = n;
    return 0;
}

/* Per-rank model-state bytes of stage 0 (plain data parallel), 1 (P_os),
 * 2 (P_os+g), 3 (P_os+g+p): fp16 params 2 B, fp16 grads 2 B and K bytes of
 * optimizer state per parameter; partitioned terms count the S = ceil(Psi/Nd)
 * parameters a rank holds.  UINT64_MAX on invalid arguments or overflow. */
uint64_t orc_model_state_bytes(uint64_t psi, uint32_t nd, uint32_t stage, uint32_t k)
{
    if (nd == 0 || stage > 3)
        return UINT64_MAX;
    uint64_t s = psi / nd + (psi % nd != 0);
    uint64_t per = 4 + (uint64_t)k;
    if (psi != 0 && per > UINT64_MAX / psi)
        return UINT64_MAX;
    switch (stage) {
    case 0: return per * psi;
    case 1: return 4 * psi + (uint64_t)k * s;
    case 2: return 2 * psi + (2 + (uint64_t)k) * s;
    default: return per * s;
    }
}

/* The same formulas with real division (Psi/Nd not rounded). */
double orc_model_state_bytes_formula(double psi, double nd, uint32_t stage, double k)
{
    switch (stage) {
    case 0: return (2 + 2 + k) * psi;
    case 1: return 4 * psi + k * psi / nd;
    case 2: return 2 * psi + (2 + k) * psi / nd;
    case 3: return (2 + 2 + k) * psi / nd;
    default: return NAN;
    }
}

/* Per-step communication volume of a data-parallel process, in parameter
 * elements, as the ZeRO summary states it (section "ZeRO-DP"): plain DP and
 * Stage 1 2*Psi (an all-reduce), Stage 2 2*Psi (reduce-scatter Psi +
 * all-gather Psi), Stage 3 3*Psi.  UINT64_MAX on an invalid stage or overflow. */
uint64_t orc_comm_volume_elems(uint64_t psi, uint32_t stage)
{
    if (stage > 3)
        return UINT64_MAX;
    uint64_t mult = stage == 3 ? 3 : 2;
    if (psi > UINT64_MAX / mult)
        return UINT64_MAX;
    return mult * psi;
}

/* Model-state bytes per GPU when ZeRO-DP (degree Nd) runs inside each of Nm
 * model-parallel slices (section "ZeRO and MP"): the slice holds ceil(Psi/Nm)
 * parameters and ZeRO partitions those over Nd. */
uint64_t orc_model_state_bytes_mp(uint64_t psi, uint32_t nd, uint32_t nm, uint32_t stage,
                                  uint32_t k)
{
    if (nm == 0)
        return UINT64_MAX;
    uint64_t slice = psi / nm + (psi % nm != 0);
    return orc_model_state_bytes(slice, nd, stage, k);
}

/* Gather of the flat range [begin, begin + len) of a partitioned buffer:
 * out[i] = element (begin + i) of the flat vector, read from the shard that
 * owns it.  Shard r's elements sit at src[r * pitch + local] (elem_bytes
 * each); S = ceil(psi / nd).  Used for the ZeRO-3 on-demand gather of a
 * layer's parameters and for resharding.  Returns -1 on a bad range. */
int orc_gather_range(const void* src, uint64_t pitch, uint64_t psi, uint32_t nd,
                     uint64_t begin, uint64_t len, uint32_t elem_bytes, void* out)
{
    if (nd == 0 || begin > psi || len > psi - begin || (elem_bytes != 2 && elem_bytes != 4))
        return -1;
    uint64_t s = psi / nd + (psi % nd != 0);
    if (s > pitch)
        return -1;
    for (uint64_t i = 0; i < len; ++i) {
        uint64_t flat = begin + i;
        uint64_t r = flat / s;
        uint64_t local = flat % s;
        const char* from = (const char*)src + (r * pitch + local) * elem_bytes;
        memcpy((char*)out + i * elem_bytes, from, elem_bytes);
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The step.                                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
    double lr, beta1, beta2, eps, weight_decay;
} orc_hparams_t;

typedef struct {
    float inv, b1, b2, c1, c2, bc1, bc2, lr, eps, wdf;
} orc_scalars_t;

/* fp32 step scalars, each formed in fp64 and rounded once. */
void orc_scalars(const orc_hparams_t* h, uint64_t t, uint32_t nd, double loss_scale,
                 orc_scalars_t* o)
{
    o->inv = (float)(1.0 / ((double)nd * loss_scale));
    o->b1 = (float)h->beta1;
    o->b2 = (float)h->beta2;
    o->c1 = (float)(1.0 - h->beta1);
    o->c2 = (float)(1.0 - h->beta2);
    o->bc1 = (float)(1.0 - pow(h->beta1, (double)t));
    o->bc2 = (float)(1.0 - pow(h->beta2, (double)t));
    o->lr = (float)h->lr;
    o->eps = (float)h->eps;
    o->wdf = (float)(1.0 - h->lr * h->weight_decay);
}

static float grad_at(const void* base, int dtype, uint64_t idx)
{
    uint16_t bits = ((const uint16_t*)base)[idx];
    return dtype == ORC_F16 ? orc_half_to_float(bits) : orc_bf16_to_float(bits);
}

/* Reduced gradient of one element: ((c_0 + c_1) + c_2) + ... + c_{Nd-1} in fp32,
 * c_j read at base[j * row_stride + idx]. */
float orc_fold(const void* base, int dtype, uint32_t nd, uint64_t row_stride, uint64_t idx)
{
    float s = grad_at(base, dtype, idx);
    for (uint32_t j = 1; j < nd; ++j)
        s = s + grad_at(base, dtype, (uint64_t)j * row_stride + idx);
    return s;
}

/* One AdamW update of one element from its scaled gradient g. */
static void adamw_elem(const orc_scalars_t* k, float g, float p, float m, float v,
                       float* p_out, float* m_out, float* v_out)
{
    /* first moment: m' = b1 * m + (1 - b1) * g */
    float m_decay = k->b1 * m;
    float m_new = k->c1 * g;
    float m1 = m_decay + m_new;
    /* second moment: v' = b2 * v + (1 - b2) * g^2 */
    float g2 = g * g;
    float v_decay = k->b2 * v;
    float v_new = k->c2 * g2;
    float v1 = v_decay + v_new;
    /* bias-corrected moments */
    float m_hat = m1 / k->bc1;
    float v_hat = v1 / k->bc2;
    /* update direction, eps outside the square root */
    float denom = sqrtf(v_hat) + k->eps;
    float u = m_hat / denom;
    /* decoupled weight decay, then the step */
    float p_decayed = p * k->wdf;
    float step = k->lr * u;
    *p_out = p_decayed - step;
    *m_out = m1;
    *v_out = v1;
}

/* The reduce-scatter of one window: out[i] = fold(i) * fp32(inv_scale) for
 * shard elements [offset, offset + n) of each row (inv_scale is given as the
 * fp32 value the caller uses).  Returns 1 if any sum is nonfinite, else 0. */
int orc_reduce_scaled(const void* grads, int dtype, uint32_t nd, uint64_t row_stride,
                      uint64_t offset, uint64_t n, float inv_scale, float* out)
{
    int flag = 0;
    for (uint64_t i = 0; i < n; ++i) {
        float s = orc_fold(grads, dtype, nd, row_stride, offset + i);
        if (!isfinite(s))
            flag = 1;
        out[i] = s * inv_scale;
    }
    return flag;
}

/* AdamW on n elements from an already reduced and scaled fp32 gradient. */
void orc_adamw_from_grad(uint64_t n, const float* g, const orc_hparams_t* h, uint64_t t,
                         const float* p, const float* m, const float* v, float* p_out,
                         float* m_out, float* v_out)
{
    orc_scalars_t k;
    orc_scalars(h, t, 1, 1.0, &k);
    for (uint64_t i = 0; i < n; ++i)
        adamw_elem(&k, g[i], p[i], m[i], v[i], &p_out[i], &m_out[i], &v_out[i]);
}

/* Unsharded data-parallel step over all Psi parameters.
 * grads: Nd rows, contributor j's gradient of element i at base[j*row_stride + i].
 * Returns 1 (and writes nothing) when any reduced sum is nonfinite; else 0,
 * with the new state in *_out and the cast parameters in params_out[0..psi). */
int orc_step_unsharded(uint64_t psi, uint32_t nd, int dtype, const void* grads,
                       uint64_t row_stride, double loss_scale, const orc_hparams_t* h,
                       uint64_t t, const float* p, const float* m, const float* v,
                       float* p_out, float* m_out, float* v_out, uint16_t* params_out)
{
    for (uint64_t i = 0; i < psi; ++i)
        if (!isfinite(orc_fold(grads, dtype, nd, row_stride, i)))
            return 1;
    orc_scalars_t k;
    orc_scalars(h, t, nd, loss_scale, &k);
    for (uint64_t i = 0; i < psi; ++i) {
        float s = orc_fold(grads, dtype, nd, row_stride, i);
        float g = s * k.inv;
        adamw_elem(&k, g, p[i], m[i], v[i], &p_out[i], &m_out[i], &v_out[i]);
        params_out[i] = dtype == ORC_F16 ? orc_float_to_half(p_out[i])
                                         : orc_float_to_bf16(p_out[i]);
    }
    return 0;
}

/* One rank's shard step, bucket by bucket through the fusion buffer cb.
 * The contribution of rank j to shard element i is base[j*row_stride + offset + i];
 * the shard's state is p/m/v[0..n); the cast parameters go to
 * params_out[slot + i].  For each bucket the reduced, scaled gradient is first
 * materialised in cb (>= min(bucket, n) floats), then the optimizer and the
 * cast run from it.  The next state is always written; the return value is 1
 * when any reduced sum of the shard was nonfinite (the caller then discards
 * the outputs on every shard), else 0. */
int orc_step_rank(uint64_t n, uint32_t nd, int dtype, const void* grads, uint64_t row_stride,
                  uint64_t offset, uint64_t bucket, float* cb, double loss_scale,
                  const orc_hparams_t* h, uint64_t t, const float* p, const float* m,
                  const float* v, float* p_out, float* m_out, float* v_out,
                  uint16_t* params_out, uint64_t slot)
{
    orc_scalars_t k;
    orc_scalars(h, t, nd, loss_scale, &k);
    int flag = 0;
    if (bucket == 0)
        return -1;
    for (uint64_t b0 = 0; b0 < n; b0 += bucket) {
        uint64_t len = n - b0 < bucket ? n - b0 : bucket;
        for (uint64_t i = 0; i < len; ++i) { /* reduce-scatter into the bucket */
            float s = orc_fold(grads, dtype, nd, row_stride, offset + b0 + i);
            if (!isfinite(s))
                flag = 1;
            cb[i] = s * k.inv;
        }
        for (uint64_t i = 0; i < len; ++i) { /* optimizer + cast from the bucket */
            uint64_t e = b0 + i;
            adamw_elem(&k, cb[i], p[e], m[e], v[e], &p_out[e], &m_out[e], &v_out[e]);
            params_out[slot + e] = dtype == ORC_F16 ? orc_float_to_half(p_out[e])
                                                    : orc_float_to_bf16(p_out[e]);
        }
    }
    return flag;
}

/* All Nd ranks' shard steps over flat state arrays (length Psi) and a gradient
 * buffer in padded-partition layout: contributor j's gradient of partition r
 * starts at grads[j * nd * pitch + r * pitch].  params_out is the flat
 * gathered buffer (rank r's slot at r*S).  Returns the OR of the ranks' flags. */
int orc_step_sharded(uint64_t psi, uint32_t nd, int dtype, const void* grads, uint64_t pitch,
                     uint64_t bucket, float* cb, double loss_scale, const orc_hparams_t* h,
                     uint64_t t, const float* p, const float* m, const float* v, float* p_out,
                     float* m_out, float* v_out, uint16_t* params_out)
{
    int flag = 0;
    for (uint32_t r = 0; r < nd; ++r) {
        uint64_t L[3];
        if (orc_layout(psi, nd, r, L) != 0)
            return -1;
        if (L[2] > pitch)
            return -1;
        int f = orc_step_rank(L[2], nd, dtype, grads, (uint64_t)nd * pitch,
                              (uint64_t)r * pitch, bucket, cb, loss_scale, h, t, p + L[1],
                              m + L[1], v + L[1], p_out + L[1], m_out + L[1], v_out + L[1],
                              params_out, L[1]);
        if (f < 0)
            return -1;
        flag |= f;
    }
    return flag;
}

/* fp64 shadow of the unsharded step (same formulas, unrounded scalars, no
 * fp32 rounding anywhere) used to bound the fp32 result.  No skip logic. */
void orc_step_unsharded_f64(uint64_t psi, uint32_t nd, int dtype, const void* grads,
                            uint64_t row_stride, double loss_scale, const orc_hparams_t* h,
                            uint64_t t, const float* p, const float* m, const float* v,
                            double* p_out, double* m_out, double* v_out)
{
    double bc1 = 1.0 - pow(h->beta1, (double)t);
    double bc2 = 1.0 - pow(h->beta2, (double)t);
    for (uint64_t i = 0; i < psi; ++i) {
        double s = 0.0;
        for (uint32_t j = 0; j < nd; ++j)
            s += (double)grad_at(grads, dtype, (uint64_t)j * row_stride + i);
        double g = s / ((double)nd * loss_scale);
        double m1 = h->beta1 * m[i] + (1.0 - h->beta1) * g;
        double v1 = h->beta2 * v[i] + (1.0 - h->beta2) * g * g;
        double u = (m1 / bc1) / (sqrt(v1 / bc2) + h->eps);
        p_out[i] = p[i] * (1.0 - h->lr * h->weight_decay) - h->lr * u;
        m_out[i] = m1;
        v_out[i] = v1;
    }
}
