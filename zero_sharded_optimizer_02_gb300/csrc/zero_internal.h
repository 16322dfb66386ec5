// Internal declarations shared by the host and device translation units of
// the ZeRO shard-step library.  Not part of the public ABI (see zero.h).
#pragma once

#include <stdint.h>

#include "zero.h"

namespace zero {

// fp32 step scalars.  Each is formed in fp64 from the caller's
// hyperparameters and rounded once to fp32, so the device arithmetic sees
// exactly these values.
struct StepScalars {
    float inv;   // 1 / (nd * loss_scale): gradient scale
    float b1;    // beta1
    float b2;    // beta2
    float c1;    // 1 - beta1
    float c2;    // 1 - beta2
    float bc1;   // 1 - beta1^t
    float bc2;   // 1 - beta2^t
    float lr;
    float eps;
    float wdf;   // 1 - lr * weight_decay
};

// Validates h (t >= 1, betas in [0,1), lr, eps, wd finite and >= 0).
bool adamw_valid(const zero_adamw_t* h);

// Scalars of step h->step; nd and loss_scale give the gradient scale
// (pass nd = 1, loss_scale = 1 when the gradient is already scaled).
StepScalars make_scalars(const zero_adamw_t* h, uint32_t nd, double loss_scale);

// Host-side validation shared by every shard-step entry point (nothing is
// launched on failure): the gradient descriptor for the shard's L->length
// elements, the in/out state (16-byte aligned; each output its input or
// disjoint from all of them), the gathered slot (2-byte aligned, no wrap,
// disjoint from the state and the rows), the flag, bucket size, loss scale
// and hyperparameters.
zero_status_t check_step_args(const zero_grads_t* g, const zero_layout_t* L,
                              const zero_state_t* in, const zero_state_t* out,
                              const void* gathered, uint64_t gathered_offset_elems,
                              uint64_t bucket_elems, double loss_scale, const zero_adamw_t* h,
                              const uint32_t* flag);

// The address the kernels access p at.  Device and managed memory are
// accessed where they are; page-locked host memory registered with CUDA is
// accessed in place over the host link (zero-copy) at its device-mapped
// address, which must share p's place within a 16-byte line; anything else
// (pageable host memory, unknown pointers) is ZERO_ERR_INVALID_ARG, since the
// GPU must not touch it; ZERO_ERR_CUDA if the runtime cannot answer (no
// device or driver).  *on_host (if given) tells whether p is host memory.
zero_status_t resolve_ptr(const void* p, void** out, bool* on_host = nullptr);

// The descriptor the kernels read: g with base replaced by the address the
// device reads it at (resolve_ptr).  *in_host (if given) tells whether the
// rows are in host memory.
zero_status_t resolve_grads(const zero_grads_t* g, zero_grads_t* out, bool* in_host = nullptr);

// True unless the environment variable ZERO_PDL (read at each call) is "0":
// step kernels, and the bucket-ready step's waits, are then launched as
// programmatic dependent launches.
bool pdl_launches();

// ZERO_OK if each of the `count` pointers is device or managed memory;
// ZERO_ERR_INVALID_ARG for host memory (pageable or page-locked) or a pointer
// CUDA does not know; ZERO_ERR_CUDA if the runtime cannot answer (no device
// or driver).  For the buffers the kernels must find in device memory: the
// fp32 state, the fusion buffer and the flag and status words.
zero_status_t require_device(const void* const* ptrs, int count);

// require_device over the six state arrays of in and out and, if non-null,
// one more word (a flag, or the gradient of the AdamW primitive).
zero_status_t require_device_state(const zero_state_t* in, const zero_state_t* out,
                                   const void* word);

// Loads now, once per device, every instance of the fused-step kernel that
// launch_fused_range can launch for `dtype` and rows where host_rows says.
// Under CUDA's lazy loading a kernel is otherwise loaded at its first
// launch, and loading can wait for kernels already running: if one of those
// is a bucket wait whose words are written only by copies the caller issues
// after this call returns, the two would wait on each other until the wait's
// time limit.
void preload_fused(int dtype, bool host_rows);

// Launches the fused step over elements [b0, b0 + len) of a shard (the
// whole shard, or one launch group of buckets) as ceil(len /
// ZERO_FUSED_WINDOW_ELEMS) launch windows of about equal length
// (for_each_window).  rows: the rows at shard element 0, at
// the address the device reads them (resolve_grads); gath: the gathered slot
// of shard element 0.  The variant follows ZERO_FUSED_VARIANT (the register
// kernel for host_rows).  gate: if non-null, every launch reads it first and
// does nothing if it is nonzero.  Returns ZERO_ERR_CUDA if a launch failed.
zero_status_t launch_fused_range(const uint16_t* rows, const zero_grads_t* g,
                                  const zero_state_t* in, const zero_state_t* out,
                                  uint16_t* gath, uint64_t b0, uint64_t len,
                                  const StepScalars& k, bool host_rows, uint32_t* d_nonfinite,
                                  const uint32_t* gate, void* stream);

}  // namespace zero
