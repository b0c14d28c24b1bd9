// tern_internal.cuh -- declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "tern.h"

namespace tern {

int sm_count();
tern_status check_matrix(const tern_matrix *w);

// Unique id of the calling thread's current CUDA context, 0 if there is none
// (keys per-context caches: a context made after a device reset is new).
unsigned long long current_context_id();

// Bound of the kernels' mbarrier waits, in SM cycles, passed to every launch
// (tern_set_wait_limit; kWaitCycles by default).
long long wait_limit();

// K == 0 products (tern_cuda.cu): y = scale * 0 (a SwiGLU pair when u != nullptr).
tern_status empty_sum(const tern_matrix *g, const tern_matrix *u, int m, float *y, cudaStream_t s);

// Tensor-core kernels (tern_mma.cu); u == nullptr means a plain projection.
tern_status gemm_mma(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int m, float *y,
                     cudaStream_t s);
tern_status take_mma_error();

// Persistent batched kernel (tern_batched.cu); items already checked.
// Number of kernel launches gemm_batched makes for these items (host only).
int batched_launches(const tern_batch_item *items, int n);
tern_status gemm_batched(const tern_batch_item *items, int n, cudaStream_t s);
// Base-3 products and unpack (arguments checked by the caller).
tern_status tern5_gemm_launch(const tern5_matrix *w, const uint16_t *x, int m, float *y, cudaStream_t s);
tern_status tern5_unpack_launch(const tern5_matrix *w, int8_t *t, cudaStream_t s);
// int8 head logits and per-row argmax (arguments checked by the caller).
tern_status head_argmax(const tern_i8_matrix *w, const uint16_t *x, int m, const float *norm_w, float eps,
                        float *logits, int32_t *argmax, cudaStream_t s);
// As gemm_batched, each item with norm_w[i] != nullptr normalised first (RMSNorm).
tern_status gemm_batched_rmsnorm(const tern_batch_item *items, const float *const *norm_w, float eps, int n,
                                 cudaStream_t s);
// As gemm_batched, with the prepared activations in a fixed module-scope
// scratch of TERN_NOALLOC_WS_BYTES (TERN_ERR_SHAPE, nothing launched, if a
// launch group needs more).
tern_status gemm_batched_noalloc(const tern_batch_item *items, int n, cudaStream_t s);
tern_status take_batched_error();

// Shared argument checks (tern_cuda.cu).
tern_status check_gemm_args(const tern_matrix *g, const tern_matrix *u, const uint16_t *x, int32_t m,
                            const float *y);

// Reads and clears every device error word (TERN_OK when all are clear).
tern_status take_device_error();

}  // namespace tern
