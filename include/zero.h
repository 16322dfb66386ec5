/*
 * zero.h -- C ABI of the ZeRO partitioned optimizer step on one GPU (sm_103a).
 *
 * One data-parallel rank of ZeRO ("ZeRO: Memory Optimizations Toward Training
 * Trillion Parameter Models", section "ZeRO-DP", Stages 1-3) owns 1/Nd of the
 * flat parameter vector.  For its shard it
 *   (1) reduces the Nd ranks' fp16/bf16 gradient contributions in fixed rank
 *       order (its half of the bucketed reduce-scatter, Stage 2), scaled by
 *       1 / (Nd * loss_scale);
 *   (2) applies mixed-precision AdamW to its fp32 master weights and Adam
 *       moments (the 4 + K bytes per parameter of section "Quantifying memory
 *       consumption", K = 12);
 *   (3) casts the new weights to fp16/bf16 into its slot of the gathered
 *       parameter buffer (the all-gather at the end of the step, Stage 1),
 * bucket by bucket (section "ZeRO-R / CB": a constant-size fusion buffer).
 * Nd ranks are emulated as Nd gradient rows in one GPU's memory.
 *
 * Conventions shared by every entry point:
 *   - Ownership: the caller owns all memory.  The library borrows the pointers
 *     for stream-ordered work and allocates nothing.  Every call is
 *     thread-safe; calls on one stream execute in order.
 *   - Pointers named d_* or documented "device" must be device (or managed)
 *     memory of the current CUDA device: the fp32 state, fusion buffers, the
 *     primitives' fp32 inputs and the flag, status and ready words.  A host
 *     pointer there (pageable or page-locked) is ZERO_ERR_INVALID_ARG before
 *     anything is launched.  Structs passed by pointer are host memory and
 *     are read before the call returns.
 *   - Gradient rows (zero_grads_t.base) and gathered parameter buffers may
 *     also be page-locked host memory registered with CUDA (cudaHostAlloc,
 *     cudaHostRegister): the kernels then read the rows, or write the cast
 *     parameters, in place over the host link at the memory's device mapping
 *     (zero-copy).  Any other host pointer, pageable memory included, is
 *     ZERO_ERR_INVALID_ARG before anything is launched.
 *   - Errors: every call validates its arguments on the host first and returns
 *     a zero_status_t without launching anything if they are invalid.  Kernel
 *     work is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream); ZERO_ERR_CUDA reports a launch error.  No exception
 *     crosses the ABI.  A nonfinite gradient is not an error: it is reported
 *     through a device flag word (see below).
 *   - Element sizes: gradients and gathered parameters are 2-byte elements
 *     (binary16 or bfloat16); optimizer state is fp32.
 *   - Arithmetic: fp32 with every operation correctly rounded and no fused
 *     multiply-add; the reduction is a sequential left fold over ranks
 *     0..Nd-1, so results do not depend on bucket size or launch shape.
 */
#ifndef ZERO_H
#define ZERO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zero_status {
    ZERO_OK = 0,
    ZERO_ERR_INVALID_ARG = 1,  /* NULL pointer, bad size, overflow, bad enum, overlap */
    ZERO_ERR_ALIGNMENT = 2,    /* a pointer or stride breaks the documented alignment */
    ZERO_ERR_CUDA = 3,         /* the CUDA runtime reported an error */
    ZERO_ERR_TIMEOUT = 4,      /* a bounded device wait expired (bucket-ready step) */
    ZERO_ERR_UNSUPPORTED = 5,  /* valid request this build does not implement */
    ZERO_ERR_IO = 6            /* a checkpoint file is missing, unreadable, torn or corrupt */
} zero_status_t;

typedef enum zero_dtype {
    ZERO_F16 = 0,   /* IEEE 754 binary16 */
    ZERO_BF16 = 1   /* bfloat16 */
} zero_dtype_t;

/* Partition of a flat buffer of psi parameters over nd ranks (ZeRO-DP: equal
 * partitions, each rank holds and updates only its own).  The last shards are
 * zero-padded: S = ceil(psi / nd), rank r owns flat indices [r*S, r*S + length). */
typedef struct zero_layout {
    uint64_t psi;          /* parameters in the flat buffer */
    uint32_t nd;           /* data-parallel degree */
    uint32_t rank;         /* this rank, 0 <= rank < nd */
    uint64_t shard_elems;  /* S = ceil(psi / nd) */
    uint64_t begin;        /* rank * S: first flat index owned (the gathered slot) */
    uint64_t length;       /* n_r = max(0, min(S, psi - begin)); 0 is a legal no-op */
    uint64_t padded_elems; /* nd * S: length of the padded flat buffer */
    uint64_t row_pitch;    /* S rounded up to row_align_elems: the emulated row pitch */
} zero_layout_t;

/* The Nd gradient contributions to one rank's shard.  The contribution of
 * rank j to shard element i is the 2-byte element
 *     base[j * row_stride + offset + i],   0 <= j < nd.
 * Full emulation (every rank's whole gradient resident): row j is rank j's
 * gradient in padded-partition layout, row_stride = nd * row_pitch,
 * offset = rank * row_pitch.  Shard view: row j holds only this shard,
 * row_stride = row_pitch, offset = 0.
 * Alignment: base 16-byte aligned; row_stride and offset multiples of 8.
 * nd: 1 <= nd <= ZERO_MAX_ND (ZERO_ERR_INVALID_ARG otherwise).
 * Memory: device (or managed) memory, or page-locked host memory registered
 * with CUDA (cudaHostAlloc, cudaHostRegister), which the kernels then read in
 * place over the host link (zero-copy: no device copy of the gradients).  Any
 * other pointer, pageable host memory included, is ZERO_ERR_INVALID_ARG
 * before anything is launched. */
/* Largest number of contribution rows a gradient descriptor may name: the
 * pages' largest data-parallel degree is 1,024; 2^24 leaves every row-count
 * computation of the kernels far from 32-bit overflow. */
#define ZERO_MAX_ND 16777216u

typedef struct zero_grads {
    const void* base;     /* device or page-locked host memory, read-only */
    uint64_t row_stride;  /* elements between consecutive ranks' rows */
    uint64_t offset;      /* element offset of this shard within every row */
    uint32_t nd;          /* number of contributions (>= 1) */
    int32_t dtype;        /* zero_dtype_t */
} zero_grads_t;

/* fp32 optimizer state of one shard, device pointers, each 16-byte aligned:
 * master weights, Adam first moment m and second moment v. */
typedef struct zero_state {
    float* master;
    float* m;
    float* v;
} zero_state_t;

/* AdamW hyperparameters (Adam with bias correction and eps outside the square
 * root; decoupled weight decay applied as p * (1 - lr * weight_decay)).  The
 * step scalars are formed in fp64 from these values and rounded once to fp32:
 * 1-beta1, 1-beta2, 1-beta1^t, 1-beta2^t, 1-lr*weight_decay. */
typedef struct zero_adamw {
    double lr;
    double beta1;         /* in [0, 1) */
    double beta2;         /* in [0, 1) */
    double eps;           /* >= 0 */
    double weight_decay;  /* >= 0 */
    uint64_t step;        /* t >= 1, the step being taken */
} zero_adamw_t;

/* Text of a status code (static storage; never NULL). */
const char* zero_status_string(zero_status_t status);

/* The ZeRO-DP partition of rank `rank` ("ZeRO-DP", Stage 1: the state is split
 * into Nd equal partitions).  row_align_elems (>= 1) rounds the emulated row
 * pitch up to a multiple (8 keeps 2-byte rows 16-byte aligned).
 * Host only.  ZERO_ERR_INVALID_ARG if out is NULL, nd == 0, rank >= nd,
 * row_align_elems == 0 or nd * S overflows. */
zero_status_t zero_partition_layout(uint64_t psi, uint32_t nd, uint32_t rank,
                                    uint32_t row_align_elems, zero_layout_t* out);

/* Per-rank model-state bytes of mixed-precision Adam ("Quantifying memory
 * consumption": fp16 params 2, fp16 grads 2, K bytes of optimizer state per
 * parameter, 16 bytes when K = 12) under stage 0 (plain data parallel),
 * 1 (P_os: 4*psi + K*S), 2 (P_os+g: 2*psi + (2+K)*S) or 3 (P_os+g+p:
 * (4+K)*S), with S = ceil(psi / nd) the parameters a rank holds; equal to
 * the pages' formulas whenever nd divides psi.  Host only.
 * Returns UINT64_MAX if nd == 0, stage > 3 or the result overflows. */
uint64_t zero_model_state_bytes(uint64_t psi, uint32_t nd, uint32_t stage, uint32_t k);

/* Reduce-scatter of one bucket (Stage 2, bucketed): for i in [0, bucket_len),
 *     s_i = (((c_0 + c_1) + c_2) + ... + c_{nd-1})   in fp32, c_j at
 *           g->base[j*row_stride + offset + bucket_begin + i],
 *     cb_out[i] = s_i * inv_scale,
 * and sets *d_nonfinite |= 1 if any s_i is inf or NaN (never clears it).
 * cb_out: device fp32[bucket_len], 4-byte aligned, the constant-size fusion
 * buffer; d_nonfinite: device uint32.  bucket_len == 0 is a no-op. */
zero_status_t zero_reduce_scatter_bucket(const zero_grads_t* g, uint64_t bucket_begin,
                                         uint64_t bucket_len, float inv_scale, float* cb_out,
                                         uint32_t* d_nonfinite, void* stream);

/* AdamW on n fp32 elements from an already reduced and scaled gradient:
 *     m' = b1 m + (1-b1) g;  v' = b2 v + (1-b2) g^2;
 *     p' = p (1 - lr wd) - lr (m'/(1-b1^t)) / (sqrt(v'/(1-b2^t)) + eps).
 * grad: device fp32[n], 4-byte aligned.  in/out state: 16-byte aligned;
 * out may equal in (in place) but may not partially overlap it. */
zero_status_t zero_adam_step_shard(const float* grad, const zero_state_t* in,
                                   const zero_state_t* out, uint64_t n,
                                   const zero_adamw_t* h, void* stream);

/* Cast of a shard's fp32 master weights into its slot of the gathered
 * parameter buffer (the local part of the Stage-1 all-gather):
 *     gathered[slot_offset_elems + i] = round_to_nearest_even(master[i]).
 * master: device fp32[n], 4-byte aligned; gathered: device or page-locked
 * host memory, 2-byte aligned (any slot phase; the store width follows it). */
zero_status_t zero_gather_params_shard(const float* master, uint64_t n, void* gathered,
                                       uint64_t slot_offset_elems, zero_dtype_t dtype,
                                       void* stream);

/* The fused shard step: reduce (1) + scale + AdamW (2) + cast into the
 * gathered slot (3) in one pass over the shard, with the reduced gradient kept in
 * registers (never materialised).  The shard length comes from L; the g->nd
 * contribution rows are folded.  g->nd is normally L->nd (Stage 2: one
 * contribution per rank) but need not be: under Stage 1 every rank holds the
 * gradient already all-reduced, so it folds a single row (g->nd = 1) and
 * passes loss_scale * Nd to keep the 1/Nd averaging.  The reduced sums stay
 * in registers, so no bucket is ever materialised and the bucket is no
 * boundary of the work: bucket_elems (>= 1) is validated but the whole shard
 * runs as ceil(n / ZERO_FUSED_WINDOW_ELEMS) launches of about equal length,
 * every cut on a 32-byte boundary of row 0 at the address the device reads
 * it (moving the cuts back to those boundaries shortens the first window and
 * can lengthen the last to ZERO_FUSED_WINDOW_ELEMS + 15 elements) (kernel boundaries keep every SM at the same place in the
 * rows; launches much longer than this let the SMs drift apart, and a cut
 * inside a 32-byte sector slows every launch after it).  A window after the
 * first starts as its predecessor drains.  Results depend on neither size.
 * The kernel is the cp.async-ring variant, except that a window that one
 * wave of the short-window kernel covers (SMs x 3 CTAs x 256 threads x 4
 * elements: 466,944 on 152 SMs) runs on that kernel (4 elements a thread,
 * so the AdamW arithmetic spreads over every SM), unless the environment
 * variable ZERO_FUSED_VARIANT, read at each call, names one kernel for every
 * window ("registers", "ring", "small" or "tma": bulk copies and
 * mbarriers); rows in host memory always use the register variant.  All
 * variants give bitwise the same results.  Launches are programmatic
 * dependent launches (each kernel waits in-kernel for its predecessor in
 * the stream, so consecutive launches lose their gap) unless the
 * environment variable ZERO_PDL is "0".
 * The new state goes to `out` and the cast parameters to
 * gathered[gathered_offset_elems + i] (device or page-locked host memory).  *d_nonfinite |= 1 if any reduced sum
 * is nonfinite; the step is then to be skipped on every shard: with out != in
 * the caller simply keeps `in` (and its previous gathered buffer).  With
 * out == in the update happens in place and cannot be rolled back: run
 * zero_check_nonfinite first.  loss_scale > 0 and finite; the gradient scale
 * is fp32(1 / (nd * loss_scale)). */
zero_status_t zero_step_shard(const zero_grads_t* g, const zero_layout_t* L,
                              const zero_state_t* in, const zero_state_t* out, void* gathered,
                              uint64_t gathered_offset_elems, uint64_t bucket_elems,
                              double loss_scale, const zero_adamw_t* h, uint32_t* d_nonfinite,
                              void* stream);

/* Bit of *d_nonfinite that a step kernel sets, besides the nonfinite bit, if
 * it gave up waiting on its own copy pipeline (a bounded wait that never
 * expires in a healthy run).  The step must then be skipped, like any nonzero
 * flag, and the caller should report ZERO_ERR_TIMEOUT. */
#define ZERO_STEP_FLAG_WAIT_TIMEOUT 0x80000000u

/* Launch-window size of the fused step, in elements: a range of n elements
 * runs as ceil(n / ZERO_FUSED_WINDOW_ELEMS) windows of about equal length,
 * none more than 15 elements longer than this (for n below 3.4e12; beyond,
 * a remainder of under 64 elements can join a full window; see
 * zero_step_shard). */
#define ZERO_FUSED_WINDOW_ELEMS 10485760ull

/* The same step unfused, through the constant-size fusion buffer: per bucket,
 * zero_reduce_scatter_bucket into cb (in the fused step's launch windows),
 * then zero_adam_step_shard from cb, then zero_gather_params_shard.  cb: device fp32 workspace of cb_elems >=
 * min(bucket_elems, L->length) + 4 elements, 16-byte aligned, owned by the
 * caller and overwritten.  Bitwise identical results to zero_step_shard. */
zero_status_t zero_step_shard_unfused(const zero_grads_t* g, const zero_layout_t* L,
                                      const zero_state_t* in, const zero_state_t* out,
                                      void* gathered, uint64_t gathered_offset_elems,
                                      uint64_t bucket_elems, double loss_scale,
                                      const zero_adamw_t* h, float* cb, uint64_t cb_elems,
                                      uint32_t* d_nonfinite, void* stream);

/* Size of the library's own fusion buffer used by zero_step_shard_unfused_static:
 * 4,194,304 fp32 values (16 MiB) of device memory in every GPU that loads the
 * library, held until the process exits.  A call needs
 * min(bucket_elems, L->length) + 4 of them, so buckets of up to
 * ZERO_STATIC_CB_MAX_BUCKET elements fit. */
#define ZERO_STATIC_CB_ELEMS 4194304ull
#define ZERO_STATIC_CB_MAX_BUCKET (ZERO_STATIC_CB_ELEMS - 4ull)

/* Allocation-free form of zero_step_shard_unfused (the paper has no
 * counterpart: this exists for callers that cannot call cudaMalloc, such as
 * a host framework whose memory pool owns the whole device and forbids
 * outside allocations, or code that must not take the device-wide
 * synchronisation that cudaMalloc/cudaFree can imply).  Same arguments and
 * results as zero_step_shard_unfused minus the workspace: the fusion buffer
 * is the library's own file-scope device array of ZERO_STATIC_CB_ELEMS
 * floats.  The caller still provides every input and output.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   - The first call on a device looks up that device's address of the array
 *     (cudaGetSymbolAddress, with the device current) and caches it with the
 *     id of the device's CUDA context.  A later call in another context of
 *     the device (after cudaDeviceReset, the array is loaded anew and may
 *     move) looks it up again.  Make the first call on a device, and the
 *     first after its context is re-created, before any stream capture.
 *   - ZERO_ERR_INVALID_ARG, with nothing launched, if
 *     min(bucket_elems, L->length) > ZERO_STATIC_CB_MAX_BUCKET; the other
 *     validation is that of zero_step_shard_unfused.
 *   - Every call on a device shares the one array and it keeps the last
 *     call's contents (nothing in it needs to start at zero: each bucket is
 *     written before it is read).  Calls whose kernels overlap on the GPU --
 *     on different streams or from different threads without ordering --
 *     race on the array and give wrong results; order them on one stream. */
zero_status_t zero_step_shard_unfused_static(const zero_grads_t* g, const zero_layout_t* L,
                                             const zero_state_t* in, const zero_state_t* out,
                                             void* gathered, uint64_t gathered_offset_elems,
                                             uint64_t bucket_elems, double loss_scale,
                                             const zero_adamw_t* h, uint32_t* d_nonfinite,
                                             void* stream);

/* Pre-pass for in-place stepping: *d_nonfinite |= 1 if any reduced sum
 * s_i (as in zero_reduce_scatter_bucket) over shard elements [begin, begin+n)
 * is nonfinite.  Reads only the gradients (2 * nd bytes per element). */
zero_status_t zero_check_nonfinite(const zero_grads_t* g, uint64_t begin, uint64_t n,
                                   uint32_t* d_nonfinite, void* stream);

/* ---- Bucket-ready stepping ------------------------------------------------- */

/* The fused step started bucket by bucket as gradients arrive ("ZeRO-DP",
 * Stage 2: gradients are reduce-scattered in buckets during the backward
 * pass).  Bucket b is elements [b*bucket_elems, ...) of the shard.
 * Consecutive buckets form launch groups: as many groups as the shard's step
 * traffic ((2*nd + 26) bytes per element) holds ZERO_STREAM_GROUP_BYTES, at
 * least one, with the buckets dealt as evenly as possible (the environment
 * variable ZERO_STREAM_GROUP_BYTES, read at each call, overrides the size: 0
 * makes every bucket its own group); for each group in order a
 * one-thread kernel waits until d_ready[b] >= epoch (wrap-around comparison)
 * for each of its buckets, then the fused step's launches for the group follow
 * on the same stream (as zero_step_shard: launch windows of about
 * ZERO_FUSED_WINDOW_ELEMS elements at most, the same choice of kernel, the
 * short-window kernel for a group that one wave of it covers).  The producer
 * of bucket b
 * writes d_ready[b] after the bucket's contributions are in place -- e.g. a
 * cudaMemcpyAsync of the word on the copy stream that copied the data.  The
 * ready words must be written by a copy engine or the host, never by a kernel
 * that would have to run concurrently with this one.  The call loads every
 * kernel it launches before its first wait starts, so that under lazy module
 * loading none of its own launches waits for that wait.
 * Each wait is bounded by timeout_ns of GPU time (%globaltimer) and an
 * iteration cap; on expiry the kernel stores ZERO_ERR_TIMEOUT into *d_status
 * (if it is still 0), touches no element of a bucket that was not seen ready,
 * and returns: the caller reads *d_status after the stream work completes.
 * timeout_ns must be in [1, ZERO_MAX_WAIT_NS] (ZERO_ERR_INVALID_ARG otherwise).
 * Other arguments, alignment and results as zero_step_shard (bitwise equal). */
#define ZERO_MAX_WAIT_NS 60000000000ull
#define ZERO_STREAM_GROUP_BYTES 1000000000ull
zero_status_t zero_step_shard_streamed(const zero_grads_t* g, const zero_layout_t* L,
                                       const zero_state_t* in, const zero_state_t* out,
                                       void* gathered, uint64_t gathered_offset_elems,
                                       uint64_t bucket_elems, double loss_scale,
                                       const zero_adamw_t* h, const uint32_t* d_ready,
                                       uint32_t epoch, uint64_t timeout_ns,
                                       uint32_t* d_nonfinite, uint32_t* d_status, void* stream);

/* Producer for zero_step_shard_streamed when the gradients come from host
 * memory: for each bucket b of the shard (elements [b*bucket_elems, ...) of
 * the first n), enqueues on copy_stream one 2D copy of the bucket's slice of
 * all nd contributor rows -- host element i of contributor j at
 * host[j * host_row_stride + i] to g's device rows -- and then a 4-byte copy
 * of *h_epoch into d_ready[b], so the ready word lands after the data.
 * host and h_epoch: pinned host memory that must stay valid and unchanged
 * until the copies complete; copy_stream must not be ordered behind the
 * stream running the consumer (use two non-blocking streams).  Only enqueues
 * copies (no kernel, no allocation).  ZERO_ERR_INVALID_ARG if a row is
 * shorter than n (host_row_stride < n, g->row_stride < g->offset + n). */
zero_status_t zero_feed_buckets(const void* host, uint64_t host_row_stride,
                                const zero_grads_t* g, uint64_t n, uint64_t bucket_elems,
                                uint32_t* d_ready, const uint32_t* h_epoch, void* copy_stream);

/* ---- ZeRO-3 parameter gather and resharding ------------------------------- */

/* On-demand gather of a flat range ("ZeRO-DP", Stage 3: parameters are
 * partitioned; a layer's are collected from their owners before use and
 * released after): out[i] = element begin + i of the flat psi-element vector,
 * for i in [0, len).  The vector is partitioned as zero_partition_layout
 * gives (S = ceil(psi / nd)); shard r's elements sit at
 * shards[r * pitch + local], local < S, pitch >= S.  elem_bytes is 2 (fp16 or
 * bf16 parameters) or 4 (fp32 state, e.g. to reshard to another nd).
 * shards and out: device memory, or page-locked host memory registered with
 * CUDA (accessed in place at its device mapping), aligned to elem_bytes;
 * any other pointer (pageable host memory) is ZERO_ERR_INVALID_ARG before
 * anything is launched.  out must not overlap the shards; only the range's
 * own elements are read.  The range spans at most
 * ceil(len / S) + 1 shard segments; one launch copies up to
 * ZERO_GATHER_SEGMENTS_PER_LAUNCH of them.  ZERO_ERR_INVALID_ARG on a range
 * outside [0, psi), pitch < S, NULL pointers or overlap. */
#define ZERO_GATHER_SEGMENTS_PER_LAUNCH 48ull
zero_status_t zero_gather_range(const void* shards, uint64_t pitch, uint64_t psi, uint32_t nd,
                                uint64_t begin, uint64_t len, uint32_t elem_bytes, void* out,
                                void* stream);

/* ---- Sharded checkpoints ---------------------------------------------------- */

/* Header of one rank's checkpoint file ("ZeRO" (process-cxr ai-library),
 * checkpointing and recovery: each rank saves only the state it owns; the
 * metadata must be stored reliably and resuming on another world size must be
 * possible).  The file is this header followed by the rank's fp32 master
 * weights, m and v, `length` elements each, in that order. */
typedef struct zero_ckpt_header {
    char magic[8];              /* "ZEROCKPT" */
    uint32_t version;           /* 2 */
    uint32_t header_bytes;      /* sizeof(zero_ckpt_header_t) */
    uint64_t psi;               /* flat parameters of the model */
    uint32_t nd;                /* data-parallel degree when saved */
    uint32_t rank;              /* the rank that saved this file */
    uint64_t shard_elems;       /* S = ceil(psi / nd) */
    uint64_t begin;             /* rank * S */
    uint64_t length;            /* elements of each array in the payload */
    uint64_t step;              /* committed optimizer steps t */
    double lr, beta1, beta2, eps, weight_decay;   /* AdamW hyperparameters */
    uint64_t payload_checksum;  /* 8-lane FNV-1a of the payload, defined below */
} zero_ckpt_header_t;

/* payload_checksum: the payload read as little-endian 32-bit words w_0,
 * w_1, ...  is split into 8 lanes (word k goes to lane k mod 8); each lane
 * runs 64-bit FNV-1a over its words, h = (h ^ w) * 0x100000001B3 from
 * h = 0xCBF29CE484222325; the checksum is 64-bit FNV-1a over the 64 bytes of
 * the 8 lane states (lane 0 first, each little-endian).  The lanes make the
 * multiply chains independent, so the sum keeps up with the file write. */

/* Writes rank L->rank's state (host fp32 arrays of L->length elements) and
 * h's hyperparameters, with h->step = the committed step count t, to `path`
 * (written to path.tmp, then renamed, so a crash leaves no torn file).
 * ZERO_ERR_INVALID_ARG on NULL arguments or a layout that
 * zero_partition_layout would not produce; ZERO_ERR_IO on a file error. */
zero_status_t zero_checkpoint_save(const char* path, const zero_layout_t* L,
                                   const zero_adamw_t* h, const float* master, const float* m,
                                   const float* v);

/* Reads and validates one file's header (magic, version, partition). */
zero_status_t zero_checkpoint_read_header(const char* path, zero_ckpt_header_t* out);

/* Loads rank L->rank of an L->nd-way partition from the n_paths files of a
 * checkpoint saved with n_paths ranks (paths[r] = old rank r's file),
 * resharding when L->nd != n_paths: the new rank's flat range is filled from
 * the overlapping ranges of the old files, so the result is bit-identical to
 * the saved state.  Every file read is checked against its payload checksum.
 * master, m, v: host arrays of L->length floats.  h_out (may be NULL)
 * receives the saved hyperparameters and step.  ZERO_ERR_INVALID_ARG if the
 * files disagree on psi or nd or are not ranks 0..n_paths-1 in order;
 * ZERO_ERR_IO on a missing, torn or corrupt file or differing steps. */
zero_status_t zero_checkpoint_load(const char* const* paths, uint32_t n_paths,
                                   const zero_layout_t* L, float* master, float* m, float* v,
                                   zero_adamw_t* h_out);

/* ---- Accounting variants ------------------------------------------------- */

/* Per-step communication volume of one data-parallel process, in parameter
 * elements, as the ZeRO summary gives it (section "ZeRO-DP"): stage 0 (plain
 * data parallel, an all-reduce) and stage 1 move 2*psi, stage 2 moves 2*psi
 * (reduce-scatter psi + all-gather psi), stage 3 moves 3*psi (1.5x).  Host
 * only.  UINT64_MAX if stage > 3 or the result overflows. */
uint64_t zero_comm_volume_elems(uint64_t psi, uint32_t stage);

/* Per-GPU model-state bytes when ZeRO-DP of degree nd runs inside each of nm
 * model-parallel slices (section "ZeRO and MP": memory falls by up to
 * Nd x Nm): zero_model_state_bytes(ceil(psi / nm), nd, stage, k).  Host only.
 * UINT64_MAX if nm == 0 or as zero_model_state_bytes. */
uint64_t zero_model_state_bytes_mp(uint64_t psi, uint32_t nd, uint32_t nm, uint32_t stage,
                                   uint32_t k);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_H */
